/*
 * kvint4.h -- C ABI of the GB300 (sm_103a) INT4 per-token-head KV cache with a
 * randomized Hadamard rotation, and of paged attention over that cache.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless it
 *   says otherwise.  The library allocates no device memory, keeps no
 *   per-call state and never synchronises the device; each call only enqueues
 *   kernels on `stream` (a cudaStream_t passed as void*; NULL is the legacy
 *   default stream) and returns.  Calls are thread-safe: host threads may
 *   call any entry point concurrently (the launch configuration each kernel
 *   needs is computed once per device and CUDA context, under a lock, and
 *   again after a cudaDeviceReset).  The one exception is
 *   kv_int4_attention_noalloc, whose calls share a device array and must not
 *   overlap on the GPU (see its note).
 * - "bf16" arguments are arrays of IEEE bfloat16 (2 bytes per element).
 * - A head vector has `head_size` = d elements; b = d & -d is the largest
 *   power-of-two divisor of d and n = d / b.  Supported head sizes: 64, 96,
 *   128, 192, 256.  Supported block size: 16.
 * - The cache layout (vLLM PR #40835, "[Feature] Triton INT4 per-token-head KV
 *   cache quantization", review thread on reshape_and_cache_per_token_head_quant):
 *     k_cache, v_cache:             uint8 [num_blocks][block_size][num_kv_heads][d/2]
 *     k_scale_cache, v_scale_cache: float [num_blocks][block_size][num_kv_heads]
 *   Slot s is (block s / block_size, offset s % block_size).  Element 2j of a
 *   head vector is the low nibble of byte j, element 2j+1 the high nibble,
 *   both signed 4-bit two's complement.
 * - Return value: KV_INT4_OK (0) or a KV_INT4_ERR_* code from host-side
 *   validation, done before anything is enqueued (on error nothing runs and
 *   no memory is touched), or KV_INT4_ERR_CUDA if a launch failed.
 * - `dev_status` (nullable) is a caller-owned device int32 that kernels OR
 *   KV_INT4_DEV_* bits into when they meet bad device-side data (an index
 *   out of range, inconsistent lengths).  The offending work is skipped; the
 *   kernels never trap or assert.  The caller clears and reads it when it
 *   chooses.
 */
#ifndef KVINT4_H
#define KVINT4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVINT4_API __attribute__((visibility("default")))
#else
#define KVINT4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* host-side status codes */
#define KV_INT4_OK 0
#define KV_INT4_ERR_NULL 1          /* a required pointer is NULL */
#define KV_INT4_ERR_HEAD_SIZE 2     /* head_size not in {64, 96, 128, 192, 256} */
#define KV_INT4_ERR_HEADS 3         /* num_q_heads % num_kv_heads != 0, a head count <= 0, or a group
                                       (num_q_heads / num_kv_heads) above 64 */
#define KV_INT4_ERR_BLOCK_SIZE 4    /* block_size != 16 */
#define KV_INT4_ERR_ALIGN 5         /* a pointer or stride breaks its alignment rule (16 bytes for
                                       K/V/Q/out and code caches, 8 for slot_mapping, 4 for scale
                                       caches and int32 metadata) */
#define KV_INT4_ERR_WORKSPACE 6     /* workspace NULL or smaller than kv_int4_attention_workspace_size() */
#define KV_INT4_ERR_SIZE 7          /* a negative count, or a size that overflows the index types */
#define KV_INT4_ERR_CUDA 8          /* a CUDA call or kernel launch failed */
#define KV_INT4_ERR_SCRATCH_LIMIT 9 /* kv_int4_attention_noalloc: the call needs more workspace than
                                       KV_INT4_NOALLOC_SCRATCH_BYTES */

/* device-side status bits (ORed into *dev_status) */
#define KV_INT4_DEV_BAD_SLOT 1      /* slot_mapping entry >= num_blocks * block_size */
#define KV_INT4_DEV_BAD_BLOCK 2     /* block_table entry outside [0, num_blocks) */
#define KV_INT4_DEV_BAD_SEQ 4       /* q_len < 0, q_len > seq_len, q_len > max_query_len,
                                       seq_len > max_blocks_per_seq * block_size, or query_start_loc
                                       outside [0, num_q_tokens] */
#define KV_INT4_DEV_BAD_SIGNS 8     /* a sign entry other than +1 / -1 */
#define KV_INT4_DEV_TIMEOUT 16      /* a wait for staged input exceeded its iteration limit: the kernel
                                       stopped early and its outputs are incomplete (not expected to occur) */

/*
 * kv_int4_write -- reshape_and_cache_int4: quantise new K/V head vectors into
 * the paged INT4 cache.
 *
 * Defined by: "Rotate KV into RHT domain in the INT4 unified attn test" (vLLM
 * PR #62881), Details / Root cause (K_s = H.D.k) and Details / Fix (rounding
 * through bf16); "vLLM -- Attention Kernels & KV Cache Quantization" (PR
 * #56198), the block-diagonal H_b for non-power-of-two d.
 *
 * For each token t < num_tokens and kv head h, with x = k[t][h][:] (and then
 * v[t][h][:]):
 *   y  = bf16_round( (I_n (x) H_b) . D . x )   H_b Sylvester Walsh-Hadamard,
 *                                              D = diag(signs), fp32 arithmetic
 *   s  = fp32(max_i |y_i| / 7)                 (0 when max|y| < 2^-120)
 *   c_i = round_half_even(y_i * fp32(1/s))     in [-7, 7] (0 when s == 0)
 * then codes go to k_cache[slot], the scale to k_scale_cache[slot] with
 * slot = slot_mapping[t].  slot < 0 marks a padding token (skipped); slot >=
 * num_blocks*block_size is skipped and sets KV_INT4_DEV_BAD_SLOT.
 *
 * k, v: bf16, element (t, h, i) at k[t*k_token_stride + h*head_size + i];
 *   heads and elements contiguous.  Strides are in elements and must be
 *   multiples of 8; k, v must be 16-byte aligned.
 * slot_mapping: int64 [num_tokens], 8-byte aligned.  signs: int8
 *   [head_size], each +1 or -1 (the random diagonal D, shared by K, V, Q and
 *   all heads).
 * Caches: as above; code caches 16-byte aligned, scale caches 4-byte
 *   aligned.  num_tokens == 0 is a no-op.
 */
KVINT4_API int kv_int4_write(const void* k, int64_t k_token_stride,
                  const void* v, int64_t v_token_stride,
                  const int64_t* slot_mapping, int num_tokens,
                  uint8_t* k_cache, uint8_t* v_cache,
                  float* k_scale_cache, float* v_scale_cache,
                  int num_blocks, int block_size, int num_kv_heads, int head_size,
                  const int8_t* signs, int32_t* dev_status, void* stream);

/*
 * kv_int4_write_prerotated -- the write path from step "s = ..." on: k and v
 * already hold the bf16 rotated values y (the rotation and the bf16 rounding
 * are skipped).  Same layout, slots and errors as kv_int4_write; no signs.
 * It exists so that codes can be compared bit for bit against an independent
 * implementation fed the same rotated values.
 */
KVINT4_API int kv_int4_write_prerotated(const void* k, int64_t k_token_stride,
                             const void* v, int64_t v_token_stride,
                             const int64_t* slot_mapping, int num_tokens,
                             uint8_t* k_cache, uint8_t* v_cache,
                             float* k_scale_cache, float* v_scale_cache,
                             int num_blocks, int block_size, int num_kv_heads, int head_size,
                             int32_t* dev_status, void* stream);

/*
 * kv_int8_write -- the int8_per_token_head sibling mode's write: quantise new
 * K/V head vectors, without rotation, into a paged int8 cache.
 *
 * Defined by: "[Feature] Triton INT4 per-token-head KV cache quantization"
 * (vLLM PR #40835), review thread (the int8 cache dtype of the per-token-head
 * modes; the raw int8 cache compared with a round reference); "vLLM --
 * Attention Kernels & KV Cache Quantization" (PR #56198), Merged
 * contribution (int8_per_token_head never uses the transform).  Per (token t,
 * kv head h) vector x of K and of V:
 *   a = max |x_i|,  s = fp32(a / 127),  c_i = rne(x_i * fp32(1 / s))  (|c_i| <= 127)
 * with s = 0 and c = 0 when a < 2^-119; c goes to cache[slot][h][:] (int8,
 * one code per element) and s to scale[slot][h].
 *
 * Arguments, ownership, slot conventions and errors are those of
 * kv_int4_write, except: k_cache / v_cache are int8 [num_blocks][block_size]
 * [num_kv_heads][head_size] (16-byte aligned), there are no signs, and
 * head_size is one of 64, 96, 128, 192, 256.
 */
KVINT4_API int kv_int8_write(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                             const int64_t* slot_mapping, int num_tokens, int8_t* k_cache, int8_t* v_cache,
                             float* k_scale_cache, float* v_scale_cache, int num_blocks, int block_size,
                             int num_kv_heads, int head_size, int32_t* dev_status, void* stream);

/*
 * kv_int4_attention_workspace_size -- bytes of device workspace that
 * kv_int4_attention needs for these sizes (a pure host computation).  The
 * workspace holds the device-built schedule, the rotated queries and the
 * split-KV partial results; its contents need no initialisation.
 * Returns 0 for invalid arguments.
 */
KVINT4_API size_t kv_int4_attention_workspace_size(int num_seqs, int num_q_tokens,
                                        int num_q_heads, int num_kv_heads, int head_size);

/*
 * kv_int4_attention -- unified_attention_int4: varlen prefill + decode
 * attention with GQA over the paged INT4 cache.
 *
 * Defined by: "Rotate KV into RHT domain in the INT4 unified attn test" (vLLM
 * PR #62881), Details / Root cause: q' = H.D.q, scores scaled by
 * softmax_scale/b so that q'.K_s/b = q.k, and D.H(.)/b applied to the output
 * to undo V's rotation; with b in place of d for block-diagonal H_b ("vLLM --
 * Attention Kernels & KV Cache Quantization", PR #56198).  Mixed batches of
 * prefills and decodes in any order ([Feature] Triton INT4 per-token-head KV
 * cache quantization, PR #40835 review thread: everything goes through
 * unified attention).
 *
 * Sequence i has query tokens [query_start_loc[i], query_start_loc[i+1]) and
 * kv length seq_lens[i] (including those tokens, whose K/V must already be in
 * the cache).  Its queries are its last q_len positions: query j sits at
 * position seq_lens[i] - q_len + j and, when `causal` != 0, sees keys
 * 0 .. that position; otherwise all seq_lens[i] keys.  With sliding_window
 * W > 0 a query at position p also sees no key at a position <= p - W (it
 * keeps the W positions ending at its own; the "added window" of the Triton
 * INT4 PR, with vLLM's window rule); W = 0 means no window and W < 0 is
 * KV_INT4_ERR_SIZE.  Blocks wholly before a sequence's window are never
 * read.  Key position p of
 * sequence i is in block block_table[i*max_blocks_per_seq + p/block_size],
 * offset p % block_size.  q head hq uses kv head hq / (num_q_heads/num_kv_heads).
 *
 * out[t][hq][:] = sum_p softmax_p(softmax_scale * q[t][hq] . k_hat_p) v_hat_p
 * with k_hat_p = D.(I_n (x) H_b).(c_p * s_p)/b the dequantised, inverse-rotated
 * key (likewise v_hat), computed in the rotated domain.
 *
 * q: bf16, element (t, hq, i) at q[t*q_token_stride + hq*head_size + i]
 *   (stride a multiple of 8 elements, 16-byte aligned).
 * out: bf16, same layout with out_token_stride.
 * block_table: int32 [num_seqs][max_blocks_per_seq].  seq_lens: int32
 *   [num_seqs].  query_start_loc: int32 [num_seqs+1], non-decreasing from 0
 *   to num_q_tokens.  These three and the scale caches are 4-byte aligned.
 *   max_query_len / max_seq_len: upper bounds of the per-sequence values
 *   (used only to size launches); a sequence whose q_len exceeds
 *   max_query_len is treated as invalid metadata (below).
 * signs: int8 [head_size], the same D that the cache was written with.
 * workspace: >= kv_int4_attention_workspace_size(...) bytes, 256-byte aligned.
 * Sequences whose metadata is invalid are skipped (their output rows are not
 * written) and set KV_INT4_DEV_BAD_SEQ; blocks outside [0, num_blocks) are
 * treated as masked and set KV_INT4_DEV_BAD_BLOCK.
 */
KVINT4_API int kv_int4_attention(const void* q, int64_t q_token_stride,
                      const uint8_t* k_cache, const uint8_t* v_cache,
                      const float* k_scale_cache, const float* v_scale_cache,
                      const int32_t* block_table, int max_blocks_per_seq,
                      const int32_t* seq_lens, const int32_t* query_start_loc,
                      int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len,
                      int num_q_heads, int num_kv_heads, int head_size,
                      int block_size, int num_blocks, float softmax_scale, int causal,
                      int sliding_window, const int8_t* signs, void* out, int64_t out_token_stride,
                      void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream);

/*
 * kv_int8_attention -- attention over the int8_per_token_head cache written
 * by kv_int8_write (the sibling mode: int8 codes of the unrotated vectors).
 *
 * Defined by: "[Feature] Triton INT4 per-token-head KV cache quantization"
 * (vLLM PR #40835), review thread (the per-token-head modes share one
 * unified attention; int8 caches); "vLLM -- Attention Kernels & KV Cache
 * Quantization" (PR #56198), Merged contribution (this mode never uses the
 * transform):
 *   out[t][hq][:] = sum_p softmax_p(softmax_scale * q[t][hq] . k_hat_p) v_hat_p,
 *   k_hat_p = c_p * s_p, v_hat_p likewise.
 * Arguments, layouts, masks (causal, sliding_window), workspace
 * (kv_int4_attention_workspace_size), device status bits and errors are
 * those of kv_int4_attention, except: k_cache / v_cache are int8
 * [num_blocks][block_size][num_kv_heads][head_size] (16-byte aligned) and
 * there are no signs.
 */
KVINT4_API int kv_int8_attention(const void* q, int64_t q_token_stride,
                                 const int8_t* k_cache, const int8_t* v_cache,
                                 const float* k_scale_cache, const float* v_scale_cache,
                                 const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                 int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len,
                                 int num_q_heads, int num_kv_heads, int head_size,
                                 int block_size, int num_blocks, float softmax_scale, int causal,
                                 int sliding_window, void* out, int64_t out_token_stride,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream);

/*
 * kv_int4_attention_noalloc -- kv_int4_attention without a caller-provided
 * workspace, for callers that cannot allocate device memory.  (The method's
 * pages have no counterpart of this entry point: it only changes where the
 * workspace lives.)
 *
 * Who needs it: code that runs inside a host framework or plugin that owns
 * all device allocations and hands it none, and pipelines whose buffers are
 * all sized up front and that must not call cudaMalloc in their steady state
 * (an allocation can synchronise the device, or fail under memory pressure).
 *
 * Arguments, layouts, results and errors are those of kv_int4_attention,
 * minus workspace and workspace_bytes.  The workspace is instead a static
 * device array of KV_INT4_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which
 * loads the library holds until the process exits.  A call whose
 * kv_int4_attention_workspace_size(...) exceeds that returns
 * KV_INT4_ERR_SCRATCH_LIMIT and enqueues nothing.  The function allocates
 * nothing (no cudaMalloc, cudaFree or allocating library call).
 *
 * The first call on a device (with that device current) looks up the array's
 * device address and keeps it (a call after a cudaDeviceReset looks it up
 * again); that call may load the library's device code on the device, so
 * make it before any stream capture begins.
 *
 * All calls on a device share the one array, which keeps the last call's
 * contents; nothing in it needs clearing (each call rewrites what it reads).
 * Calls whose work overlaps on the GPU -- different streams, or host threads
 * without ordering -- race on the array and give wrong results: order them,
 * e.g. by issuing them on one stream.
 */
#define KV_INT4_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
KVINT4_API int kv_int4_attention_noalloc(const void* q, int64_t q_token_stride,
                                         const uint8_t* k_cache, const uint8_t* v_cache,
                                         const float* k_scale_cache, const float* v_scale_cache,
                                         const int32_t* block_table, int max_blocks_per_seq,
                                         const int32_t* seq_lens, const int32_t* query_start_loc,
                                         int num_seqs, int num_q_tokens, int max_query_len, int max_seq_len,
                                         int num_q_heads, int num_kv_heads, int head_size,
                                         int block_size, int num_blocks, float softmax_scale, int causal,
                                         int sliding_window, const int8_t* signs, void* out,
                                         int64_t out_token_stride, int32_t* dev_status, void* stream);

/*
 * In-slot scale layout: K, V, codes and scales in one cache tensor.
 *
 * Defined by: "[Feature] Triton INT4 per-token-head KV cache quantization"
 * (vLLM PR #40835), review thread (the cache-layout diff: a block holds a K
 * half then a V half; every (token, head) slot is padded_hs wide with the f32
 * scale at offset hs inside it) and "Rotate KV into RHT domain in the INT4
 * unified attn test" (PR #62881), Validation (#62113: 16-byte-aligned
 * per-token-head KV slots).  Reading taken: with CB code bytes per head
 * vector (head_size / 2 for INT4, head_size for int8) a slot is
 *   P = kv_int4_inslot_slot_bytes(head_size, int8) = round_up(CB + 4, 16) bytes:
 * codes at [0, CB), the f32 scale at [CB, CB + 4), padding after (CB is a
 * multiple of 16, so the scale and the padding are the slot's last 16
 * bytes: a write stores them together, the scale then zeros, so that it
 * writes whole DRAM sectors; attention never reads the padding, and the
 * padding of slots no write touches keeps its bytes); the cache is uint8
 * [num_blocks][2 (K, V)][block_size]
 * [num_kv_heads][P], 16-byte aligned: the codes of token slot s, kv head h,
 * half kv (0: K, 1: V) start at byte
 *   (((s / 16) * 2 + kv) * 16 + s % 16) * num_kv_heads * P + h * P
 * and its scale CB bytes further on.
 *
 * The writes and attentions below are kv_int4_write / kv_int8_write and
 * kv_int4_attention / kv_int8_attention with the four cache and scale
 * pointers replaced by that one tensor; everything else is identical.
 * kv_int4_inslot_slot_bytes returns 0 for an unsupported head size.
 */
KVINT4_API int kv_int4_inslot_slot_bytes(int head_size, int int8);
KVINT4_API int kv_int4_write_inslot(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                                    const int64_t* slot_mapping, int num_tokens, uint8_t* kv_cache, int num_blocks,
                                    int block_size, int num_kv_heads, int head_size, const int8_t* signs,
                                    int32_t* dev_status, void* stream);
KVINT4_API int kv_int8_write_inslot(const void* k, int64_t k_token_stride, const void* v, int64_t v_token_stride,
                                    const int64_t* slot_mapping, int num_tokens, uint8_t* kv_cache, int num_blocks,
                                    int block_size, int num_kv_heads, int head_size, int32_t* dev_status,
                                    void* stream);
KVINT4_API int kv_int4_attention_inslot(const void* q, int64_t q_token_stride, const uint8_t* kv_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
                                        int num_q_tokens, int max_query_len, int max_seq_len, int num_q_heads,
                                        int num_kv_heads, int head_size, int block_size, int num_blocks,
                                        float softmax_scale, int causal, int sliding_window, const int8_t* signs,
                                        void* out, int64_t out_token_stride, void* workspace,
                                        size_t workspace_bytes, int32_t* dev_status, void* stream);
KVINT4_API int kv_int8_attention_inslot(const void* q, int64_t q_token_stride, const uint8_t* kv_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
                                        int num_q_tokens, int max_query_len, int max_seq_len, int num_q_heads,
                                        int num_kv_heads, int head_size, int block_size, int num_blocks,
                                        float softmax_scale, int causal, int sliding_window, void* out,
                                        int64_t out_token_stride, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_status, void* stream);

/*
 * kv_int4_rht -- the block-diagonal randomized Hadamard rotation on its own:
 * the rotation the write path applies to K and V before quantising them (the
 * pages' single_rht step), and its inverse.
 *
 * Defined by: "vLLM -- Attention Kernels & KV Cache Quantization" (PR
 * #56198), Merged contribution: with b the largest power-of-two divisor of
 * head_size d and n = d / b, H_b (unnormalised Sylvester Walsh-Hadamard,
 * H_b H_b^T = b I) acts on each of the n contiguous blocks of b elements;
 * "Rotate KV into RHT domain in the INT4 unified attn test" (PR #62881),
 * Details / Root cause: the random +-1 diagonal D is applied first.
 *
 *   inverse == 0:  y = (I_n (x) H_b) . D . x
 *   inverse != 0:  y = D . (I_n (x) H_b) . x / b      (so rht(rht(x), inverse) = x)
 *
 * Arithmetic in fp32 (one rounding per butterfly stage); the result is
 * stored as bf16 (round to nearest even) or, with y_f32 != 0, as fp32.  Any
 * head_size in [1, 4096] (odd d gives b = 1: y = D x, resp. D y).
 *
 * x        device, bf16 [num_rows][head_size], row stride x_row_stride
 *          elements (>= head_size), 2-byte aligned
 * y        device, [num_rows][head_size] bf16 (y_f32 == 0) or fp32, row
 *          stride y_row_stride elements (>= head_size), naturally aligned;
 *          must not overlap x
 * signs    device, int8 [head_size], entries +1 / -1 (anything < 0 counts as -1)
 * stream   a cudaStream_t (NULL: the legacy default stream)
 *
 * Returns KV_INT4_OK after enqueueing one kernel (nothing for num_rows == 0),
 * KV_INT4_ERR_NULL for a NULL x, y or signs with num_rows > 0,
 * KV_INT4_ERR_HEAD_SIZE for head_size outside [1, 4096], KV_INT4_ERR_ALIGN
 * for a misaligned pointer or a row stride below head_size, KV_INT4_ERR_SIZE
 * for num_rows < 0, KV_INT4_ERR_CUDA if the launch failed.
 */
KVINT4_API int kv_int4_rht(const void* x, int64_t x_row_stride, void* y, int64_t y_row_stride, int y_f32,
                           int64_t num_rows, int head_size, const int8_t* signs, int inverse, void* stream);

/*
 * Kernel timing for benchmarks (off by default, per host thread; not part of
 * the method).  While enabled on the calling thread, every kv_int4_write and
 * kv_int4_attention call records a pair of CUDA events on its stream around
 * each of its kernels.  kv_int4_timing_collect waits for the recorded events
 * and writes, per kernel kind, the summed device time in ms, the number of
 * timed launches and the number of launches that could not be timed (more
 * than 4096 pending, or an event error); then it clears the record.  Arrays
 * have KV_INT4_TIMED_KINDS entries, in the order KV_INT4_TIMED_*.  Any
 * pointer may be NULL.  Returns KV_INT4_ERR_CUDA if an event query failed.
 */
#define KV_INT4_TIMED_KINDS 5
#define KV_INT4_TIMED_WRITE 0    /* the write kernel */
#define KV_INT4_TIMED_PREP 1     /* attention: schedule + query rotation */
#define KV_INT4_TIMED_PREFILL 2  /* attention: prefill tiles */
#define KV_INT4_TIMED_DECODE 3   /* attention: split-KV decode */
#define KV_INT4_TIMED_REDUCE 4   /* attention: split merge + inverse rotation */
KVINT4_API int kv_int4_timing_enable(int enable);
KVINT4_API int kv_int4_timing_collect(double* ms, int* launches, int* dropped);

/* kv_int4_status_string -- a static, human-readable name for a KV_INT4_* code. */
KVINT4_API const char* kv_int4_status_string(int status);

/* kv_int4_selftest_wait -- self-test of the bounded barrier wait that the pipelined kernels use
 * (the write kernel's copy stages, the prefill's hand-offs between warp roles): one warp waits on
 * an mbarrier that nothing arrives at, gives up after `iterations` attempts, ORs
 * KV_INT4_DEV_TIMEOUT into *dev_status and returns; the SM cycles it waited go to *dev_cycles
 * (nullable).  It never faults or hangs: it exercises the time-out path on a GPU, and its cycles
 * per attempt bound how long the kernels' own limit (2^18 attempts, about a second) can hold a
 * warp.  Device pointers, enqueued on `stream` (a cudaStream_t passed as void*).  KV_INT4_ERR_SIZE for iterations < 0,
 * KV_INT4_ERR_NULL without dev_status. */
KVINT4_API int kv_int4_selftest_wait(int iterations, int32_t* dev_status, uint64_t* dev_cycles,
                                     void* stream);

/* kv_int4_version -- the library's ABI version: 4 (2: kv_int4_rht and the int8_per_token_head
 * entry points kv_int8_write / kv_int8_attention, sliding_window in the attention entry points;
 * 3: the in-slot entry points, kv_int4_attention_noalloc's window argument, kv_int4_selftest_wait;
 * 4: kv_int4_selftest_wait takes its stream as void*, like every other entry point). */
KVINT4_API int kv_int4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVINT4_H */
