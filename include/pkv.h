/*
 * pkv — paged KV cache and decode attention for one GB300 (sm_103a).
 *
 * Plain C ABI: opaque handles, raw pointers, sizes and status codes.  No C++ or
 * framework types cross it and no exception leaves it.  Pointers documented as
 * "device" must be CUDA device (or managed) memory on the pool's device; "host"
 * pointers are ordinary CPU memory.  The caller owns every buffer it passes; the
 * pool owns its own device storage.  Kernels run asynchronously on the caller's
 * stream (NULL = the legacy default stream); argument errors are reported
 * synchronously and launch nothing.  Faults that only the device can see (a
 * block id or slot outside the pool, an over-long context) are recorded in the
 * pool's device error word and read back with pkv_check_device_error(); the
 * kernels never read or write outside the pool or the caller's buffers.
 *
 * Nothing here is thread-safe: serialise calls that touch the same pool or
 * allocator.
 *
 * Problem statement (page title, section):
 *  - "TensorRT-LLM 深度实战" (chenxutan.com), §3.1 Paged KV Cache: the KV memory is
 *    cut into fixed pages, handed to sequences on demand from a free-page list
 *    and returned when a sequence finishes; a per-sequence page table maps a
 *    sequence to its pages.
 *  - "TensorRT-LLM 推理加速实战" (socake.github.io), §8 KV Cache 深入: block_size 64
 *    (vLLM uses 16); FP8 KV cache (fp8_e4m3); §8.1 the KV bytes-per-token formula;
 *    §7.2 masked_mha, the decode-phase attention of one new token per request.
 *  - "TensorRT-LLM加速大模型推理实战" (codearts.csdn.net): GQA/MQA, several query
 *    heads sharing one KV head.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_pool pkv_pool;
typedef struct pkv_allocator pkv_allocator;
/* Same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* bad size, null or misaligned pointer, unsupported shape */
    PKV_ERR_OOM = 2,         /* not enough free blocks (nothing was changed) or cudaMalloc failed */
    PKV_ERR_NO_SEQ = 3,      /* unknown sequence id */
    PKV_ERR_BOUNDS = 4,      /* index outside the pool / table / capacity (host check or device flag) */
    PKV_ERR_CUDA = 5,        /* a CUDA runtime call failed */
    PKV_ERR_TIMEOUT = 6      /* a kernel's bounded wait ran out (device flag); results are invalid */
} pkv_status;

typedef enum {
    PKV_KV_BF16 = 0,      /* K/V stored as bf16 */
    PKV_KV_FP8_E4M3 = 1,  /* K/V stored as OCP E4M3 codes with one fp32 scale per (block, K|V, head) */
    PKV_KV_INT8 = 2       /* K/V stored as int8 codes in [-127, 127], same scale layout (amax / 127) */
} pkv_dtype;

/* ------------------------------------------------------------------ block allocator (host)
 * The pages' PagedKVCache ("TensorRT-LLM 深度实战", §3.1): a free list that starts as
 * 0..num_blocks-1 and hands out blocks with pop() from its end, a table
 * seq_id -> [block ids] in the order the blocks were taken, growth by whole
 * blocks, and release that appends a sequence's blocks back in table order.
 * Unlike the page's sketch, running out of blocks changes nothing.
 */

/* num_blocks >= 1; block_size a power of two in [16, 256].  *out is owned by the caller
 * and freed with pkv_allocator_destroy. */
pkv_status pkv_allocator_create(int num_blocks, int block_size, pkv_allocator** out);
pkv_status pkv_allocator_destroy(pkv_allocator* a);

/* Replace the free list by order[0..n) (the last entry is handed out first).  Only while
 * no sequence holds blocks; order must be a permutation of 0..num_blocks-1. */
pkv_status pkv_allocator_set_free_order(pkv_allocator* a, const int32_t* order_host, int n);

/* Shuffle the current free list in place with a seeded Fisher-Yates (Durstenfeld) pass: for
 * i = n-1 down to 1, swap entries i and j, where the k-th swap (k = 0, 1, ...) takes
 * j = ((x_k >> 11) * (i + 1)) >> 53 and x_k is the k-th output of splitmix64 started from `seed`
 * (x_k = mix(seed + (k + 1) * 0x9E3779B97F4A7C15), mix: z ^= z >> 30, z *= 0xBF58476D1CE4E5B9,
 * z ^= z >> 27, z *= 0x94D049BB133111EB, z ^= z >> 31).  On a fresh allocator the list becomes
 * that permutation of 0..num_blocks-1 (a seeded, fragmented allocation order for tests and
 * benchmarks, "TensorRT-LLM 深度实战" §3.1's free-page list); blocks held by sequences are not
 * affected.  Deterministic and identical on every platform. */
pkv_status pkv_allocator_shuffle_free_list(pkv_allocator* a, uint64_t seed);

/* Make seq_id able to hold n_tokens tokens: an unknown seq_id is created with
 * ceil(n_tokens / block_size) blocks, a known one takes ceil((n_tokens - capacity) /
 * block_size) more when n_tokens exceeds its capacity.  PKV_ERR_OOM if the free list is
 * too short; then neither the sequence nor the free list changes. */
pkv_status pkv_seq_reserve(pkv_allocator* a, int64_t seq_id, int64_t n_tokens);

/* pkv_seq_reserve for count sequences in order (one decode step grows every running sequence
 * by a token).  Stops at the first failure: returns its status and, in *done, how many
 * reservations succeeded (those stay in place). */
pkv_status pkv_seq_reserve_many(pkv_allocator* a, const int64_t* seq_ids_host, const int64_t* n_tokens_host,
                                int64_t count, int64_t* done);

/* Drop seq_id: each of its blocks loses one holder, and blocks left with none are appended to
 * the free list in table order.  Forgets seq_id. */
pkv_status pkv_seq_release(pkv_allocator* a, int64_t seq_id);

/* Block reuse (the pages' enable_block_reuse / enable_kv_cache_reuse: a new request reuses the
 * KV blocks of a cached prefix, "TensorRT-LLM 推理加速实战" §8).  New sequence dst_seq starts with
 * the first n_tokens tokens of src_seq: src's first n_tokens / block_size blocks are shared
 * (each gains a holder).  If n_tokens ends inside a block, dst gets a fresh block for it and
 * *cow_src_block / *cow_dst_block name the block to copy (pkv_pool_copy_block) before dst
 * appends; otherwise both are -1.  Appends to dst must start at position n_tokens, so no
 * shared block is ever written.  PKV_ERR_NO_SEQ (src unknown), PKV_ERR_INVALID_ARG (dst exists
 * or equals src), PKV_ERR_BOUNDS (n_tokens beyond src's capacity), PKV_ERR_OOM (no block for the
 * copy); on error nothing changes. */
pkv_status pkv_seq_share_prefix(pkv_allocator* a, int64_t src_seq, int64_t dst_seq, int64_t n_tokens,
                                int32_t* cow_src_block, int32_t* cow_dst_block);

/* Number of sequences holding `block` (0 = on the free list). */
pkv_status pkv_block_refcount(const pkv_allocator* a, int32_t block, int* out);

/* Number of blocks seq_id holds (PKV_ERR_NO_SEQ if unknown). */
pkv_status pkv_seq_num_blocks(const pkv_allocator* a, int64_t seq_id, int* out);

pkv_status pkv_num_free_blocks(const pkv_allocator* a, int* out);

/* Copy the free list (index n-1 is handed out next) into out_host[0..capacity); *n gets its
 * length.  PKV_ERR_BOUNDS if capacity is too small (nothing written). */
pkv_status pkv_free_list(const pkv_allocator* a, int32_t* out_host, int capacity, int* n);

/* Pack the block tables of seq_ids[0..B) into out_host[B][max_blocks] (int32, row-major),
 * padding with -1.  PKV_ERR_NO_SEQ for an unknown id, PKV_ERR_BOUNDS if a sequence holds
 * more than max_blocks blocks. */
pkv_status pkv_get_block_tables(const pkv_allocator* a, const int64_t* seq_ids_host, int B, int max_blocks,
                                int32_t* out_host);

/* out_host[i] = table(seq_ids[i])[pos / block_size] * block_size + pos % block_size for
 * pos = positions[i]; a negative position gives -1 (a padding token that pkv_append skips).
 * PKV_ERR_BOUNDS if a position is beyond the sequence's capacity. */
pkv_status pkv_slot_mapping(const pkv_allocator* a, const int64_t* seq_ids_host, const int64_t* positions_host,
                            int64_t N, int64_t* out_host);

/* Host inputs of one step in one call (the bookkeeping of an in-flight batching step, page
 * "TensorRT-LLM 深度实战" §3.2, §7.3), equal to the composition of the calls above.
 *
 * pkv_stage_prefill: a chunked prefill call of n sequences, sequence i prefilling positions
 * p0[i] .. p1[i]-1.  In order, every sequence is grown to hold p1[i] tokens (pkv_seq_reserve;
 * stops at the first failure, earlier reservations stay), then written: tables_out
 * [n][max_blocks] (pkv_get_block_tables), slots_out [sum(p1 - p0)] the chunk rows' slots packed
 * sequence after sequence, cu_out [n + 1] the packed offsets (cu_out[0] = 0) and ctx_out [n] =
 * p1.  Caller-owned host buffers of at least those sizes.  PKV_ERR_INVALID_ARG (nothing changed)
 * when p0 < 0, p1 < p0, a count or position exceeds int32 or max_blocks < 1; otherwise the
 * status of the failing reservation or table write. */
pkv_status pkv_stage_prefill(pkv_allocator* a, const int64_t* seq_ids_host, const int64_t* p0_host,
                             const int64_t* p1_host, int n, int max_blocks, int64_t* slots_out_host,
                             int32_t* cu_out_host, int32_t* ctx_out_host, int32_t* tables_out_host);

/* pkv_stage_decode: one decode step of n sequences, sequence i appending its token at position
 * pos[i].  In order, every sequence is grown to hold pos[i] + 1 tokens (as above), then written:
 * tables_out [n_pad][max_blocks], slots_out [n_pad] (the slot of position pos[i]) and lens_out
 * [n_pad] = pos[i] + 1; rows n .. n_pad-1 are padding (table row -1, slot -1, length 0), as a
 * batch-size bucket of a captured step needs.  PKV_ERR_INVALID_ARG (nothing changed) when
 * n_pad < n, pos < 0 or pos + 1 exceeds int32. */
pkv_status pkv_stage_decode(pkv_allocator* a, const int64_t* seq_ids_host, const int64_t* pos_host, int n, int n_pad,
                            int max_blocks, int32_t* tables_out_host, int64_t* slots_out_host, int32_t* lens_out_host);

/* ------------------------------------------------------------------ pool (device)
 * Device layout ("block pool"): block b, K (kv=0) or V (kv=1), KV head h form one
 * contiguous tile of block_size*head_dim elements starting at element
 * ((b*2 + kv)*n_kv_heads + h) * block_size * head_dim.
 *   bf16 K and V, fp8 K:  row-major [block_size][head_dim] (token t, dim d at t*D + d).
 *   fp8 V: block_size/16 panels of [head_dim][16]: (t, d) at (t/16)*D*16 + d*16 + pos(t%16),
 *   each 16-byte panel row holding its tokens in the order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15
 *   (so one 4-byte load yields the token pairs one MMA k-step consumes).
 *   fp8 scales: float[num_blocks][n_kv_heads][4]; [..][0] scales K, [..][1] scales V,
 *   [..][2..3] are zero padding (one 16-byte record per block and head).
 * An element's value is bf16(bits) or e4m3(code) * scale.
 */

/* head_dim 64 or 128; block_size a power of two in [16, 256]; n_kv_heads >= 1.  Allocates
 * the pool with cudaMalloc on the current device and zero-fills it; the pool embeds an
 * allocator over the same num_blocks (see pkv_pool_allocator). */
pkv_status pkv_pool_create(int num_blocks, int block_size, int n_kv_heads, int head_dim, pkv_dtype kv_dtype,
                           pkv_pool** out);
pkv_status pkv_pool_destroy(pkv_pool* pool);

/* The pool's own allocator; owned by the pool (do not destroy it). */
pkv_status pkv_pool_allocator(pkv_pool* pool, pkv_allocator** out);

/* Raw device buffers for inspection: the KV bytes and the fp8 scale array (NULL and 0 for
 * bf16 pools).  Ownership stays with the pool. */
pkv_status pkv_pool_raw(const pkv_pool* pool, void** kv_dev, size_t* kv_bytes, float** scales_dev,
                        size_t* scale_bytes);

/* Copy block src_block's K and V (every head) and, for fp8 pools, its scale records onto
 * dst_block, asynchronously on `stream` (the copy-on-write step of pkv_seq_share_prefix). */
pkv_status pkv_pool_copy_block(pkv_pool* pool, int32_t src_block, int32_t dst_block, pkv_stream_t stream);

/* Synchronise the device, read and clear the pool's device error word.  Returns PKV_OK,
 * PKV_ERR_BOUNDS (a kernel saw an out-of-range block id, slot or context length and
 * skipped or clamped it) or PKV_ERR_TIMEOUT (a bounded wait expired). */
pkv_status pkv_check_device_error(pkv_pool* pool);

/* ------------------------------------------------------------------ append (device)
 * Write each new token's K and V into its physical slot ("TensorRT-LLM 深度实战", §3.1
 * append_tokens, whose pages hold the tokens' K/V).
 *   k_new_dev, v_new_dev: bf16 [N][n_kv_heads][head_dim], 16-byte aligned.
 *   slot_mapping_dev: int64 [N]; slot = block * block_size + offset; -1 skips the token.
 * bf16 pools store the bits.  fp8 pools quantise: for every (block, K|V, head) whose offset 0
 * this call writes, the scale becomes amax/448 over this call's tokens in that block (1 if
 * the amax is 0); other blocks keep their stored scale; each value is stored as
 * e4m3_rne_satfinite(x / scale) with an IEEE fp32 division.  A slot beyond the pool is
 * skipped and flagged (PKV_ERR_BOUNDS via pkv_check_device_error).  Two tokens of one call
 * must not share a slot.  Calls that overlap in time on one pool race. */
pkv_status pkv_append(pkv_pool* pool, const void* k_new_dev, const void* v_new_dev, const int64_t* slot_mapping_dev,
                      int64_t N, pkv_stream_t stream);

/* ------------------------------------------------------------------ RoPE fused into the append
 * "TensorRT-LLM 深度实战", §3.3-3.4: RoPE is fused with the attention's neighbouring kernels
 * (use_fused_rope).  Rotary position embedding in the Llama "rotate half" form: element d of the
 * first half of a row pairs with d + D/2 and, at position p, the pair turns by the angle
 * p * rope_base^(-2d/D):  y[d] = x[d] cos - x[d+D/2] sin,  y[d+D/2] = x[d+D/2] cos + x[d] sin.
 * Angle, cosine, sine and rotation are computed in fp64 and rounded to bf16 (nearest, ties to
 * even) once.
 *   k_new_dev: bf16 [N][n_kv_heads][head_dim], rotated IN PLACE at positions_dev, then appended
 *     like pkv_append (bf16 pools: the rotation and the scatter are one kernel; fp8 pools: the
 *     rotated rows then go through the quantising append).
 *   v_new_dev, slot_mapping_dev: as pkv_append.
 *   positions_dev: int64 [N], the tokens' positions in their sequences (>= 0).
 *   q_dev: optional bf16 [N][n_q_heads][head_dim] (the same tokens' queries), rotated in place
 *     with the same positions; NULL to skip.
 *   rope_base: > 1 and finite (10000 for Llama-2, 500000 for Llama-3).
 * Errors as pkv_append; PKV_ERR_INVALID_ARG for a bad base, positions or q. */
pkv_status pkv_append_rope(pkv_pool* pool, void* k_new_dev, const void* v_new_dev, const int64_t* slot_mapping_dev,
                           const int64_t* positions_dev, int64_t N, double rope_base, void* q_dev, int n_q_heads,
                           pkv_stream_t stream);

/* ------------------------------------------------------------------ decode attention (device)
 * For each sequence b and query head j, with KV head h = j / (n_q_heads / n_kv_heads):
 *   out[b][j] = softmax_t(scale * <q[b][j], K_b[t]>) . V_b[t],  t < context_lens[b],
 * K_b/V_b[t] read from block block_tables[b][t / block_size] at offset t % block_size
 * ("TensorRT-LLM 推理加速实战", §7.2 masked_mha).  Work is split over the context in 64-token
 * groups balanced across the GPU; partial softmax states (running max, sum, weighted V)
 * of a sequence cut between CTAs are merged with the log-sum-exp rule.
 *   q_dev: bf16 [B][n_q_heads][head_dim], 16-byte aligned.
 *   block_tables_dev: int32 [B][max_blocks]; context_lens_dev: int32 [B].
 *   out_dev: bf16 [B][n_q_heads][head_dim], 16-byte aligned (fp32 accumulation, RNE to bf16).
 *   workspace_dev: >= pkv_decode_workspace_bytes() bytes, 256-byte aligned, zero-filled
 *   before its first use (pkv_decode_workspace_init); every call leaves it ready for the
 *   next.  Calls that overlap in time must use different workspaces.
 * n_q_heads must be a multiple of n_kv_heads with at most 8 query heads per KV head.
 * context_lens[b] == 0 yields zeros.  A context longer than max_blocks*block_size, or a
 * block id outside the pool, is clamped/skipped and flagged (PKV_ERR_BOUNDS).  Every wait in
 * the kernel is bounded (2 s); if one runs out the results are invalid, pkv_check_device_error
 * returns PKV_ERR_TIMEOUT, and the workspace must be re-initialised before its next use. */
pkv_status pkv_decode_attention(const pkv_pool* pool, const void* q_dev, const int32_t* block_tables_dev,
                                int max_blocks, const int32_t* context_lens_dev, int B, int n_q_heads, float scale,
                                void* out_dev, void* workspace_dev, size_t workspace_bytes, pkv_stream_t stream);

/* ------------------------------------------------------------------ decode step (device)
 * One step of in-flight batching for one layer ("TensorRT-LLM 深度实战", §3.2: every step the
 * running batch appends one token per sequence and runs one forward pass): pkv_append of the
 * step's new K/V followed by pkv_decode_attention over the grown contexts.  Same arguments,
 * layouts, results and errors as those two calls made in sequence; all arguments are checked
 * before anything is launched.  On a bf16 pool (and for more than 1024 new tokens) the
 * attention kernel is launched as a programmatic dependent of the append, so its set-up
 * (context lengths, block tables, query rows) overlaps the append and its first pool read waits
 * for the append to finish — the per-step launch overhead the pages counter with CUDA graphs
 * ("TensorRT-LLM 推理加速实战", §7.1).  On an FP8 or INT8 pool with 1 to 1024 new tokens one
 * kernel does both: its warps quantise the new rows (the same codes and scales as pkv_append)
 * while its set-up runs, and every page and scale is read after all rows are in.  That launch is
 * cooperative (all its CTAs resident at once, which a GPU busy with other work can delay) and
 * uses 33 words of the workspace (32 item counters 128 bytes apart and a CTA count, about 4 KB,
 * included in pkv_decode_workspace_bytes), which return to zero like the merge tickets; its wait is
 * bounded like the others.  The append must not write q, block_tables or context_lens (it only
 * writes the pool). */
pkv_status pkv_decode_step(pkv_pool* pool, const void* k_new_dev, const void* v_new_dev,
                           const int64_t* slot_mapping_dev, int64_t N, const void* q_dev,
                           const int32_t* block_tables_dev, int max_blocks, const int32_t* context_lens_dev, int B,
                           int n_q_heads, float scale, void* out_dev, void* workspace_dev, size_t workspace_bytes,
                           pkv_stream_t stream);

/* pkv_decode_step with RoPE fused into its append (pkv_append_rope): the step's new K rows and
 * query rows are rotated at positions_dev (in place, k_new_dev and q_dev), K/V appended, then
 * the attention runs over the grown contexts as a programmatic dependent of the append; it
 * reads q only after the append has finished.  N must equal B (one new token per sequence). */
pkv_status pkv_decode_step_rope(pkv_pool* pool, void* k_new_dev, const void* v_new_dev,
                                const int64_t* slot_mapping_dev, const int64_t* positions_dev, int64_t N,
                                double rope_base, void* q_dev, const int32_t* block_tables_dev, int max_blocks,
                                const int32_t* context_lens_dev, int B, int n_q_heads, float scale, void* out_dev,
                                void* workspace_dev, size_t workspace_bytes, pkv_stream_t stream);

/* Workspace size for pkv_decode_attention and pkv_decode_step with these B, n_q_heads and
 * max_blocks. */
pkv_status pkv_decode_workspace_bytes(const pkv_pool* pool, int B, int n_q_heads, int max_blocks, size_t* out);

/* cudaMemsetAsync(workspace, 0, bytes, stream): prepares a fresh workspace. */
pkv_status pkv_decode_workspace_init(void* workspace_dev, size_t workspace_bytes, pkv_stream_t stream);

/* ------------------------------------------------------------------ prefill (chunked context)
 * Chunked-context attention over the pool: "TensorRT-LLM 深度实战", §7.3 (a long input is
 * processed chunk by chunk, each chunk interleaved with decode steps) and "TensorRT-LLM 推理
 * 加速实战", §7.2 (context_fmha, the prefill attention; use_paged_context_fmha reads the paged
 * cache).  Sequence b's chunk is the query rows cu_q_lens[b] .. cu_q_lens[b+1]-1; its K/V have
 * already been appended, so its cache holds context_lens[b] tokens of which the chunk's
 * n_b = cu_q_lens[b+1]-cu_q_lens[b] are the last.  Query i of the chunk sits at position
 * context_lens[b] - n_b + i and attends causally to the cached tokens 0 .. that position:
 *     out[row][j] = sum_{t <= pos} softmax_t(scale * q[row][j] . K_b[t]) V_b[t],
 * query head j reading KV head j / (n_q_heads / n_kv_heads).
 *   q_dev, out_dev: bf16 [cu_q_lens[B]][n_q_heads][head_dim], 16-byte aligned (rows of all chunks
 *     packed back to back); fp32 accumulation, output rounded to bf16 (RNE).
 *   cu_q_lens_dev: int32 [B+1], non-decreasing, cu_q_lens[0] = 0.
 *   max_q_len: host int >= every n_b (sizes the grid; 0 launches nothing).
 *   block_tables_dev: int32 [B][max_blocks]; context_lens_dev: int32 [B].
 * Pools: bf16, FP8-E4M3 or INT8.  On a one-byte pool the tensor-core products run in f16: K's
 * codes exactly (their (block, head) scale multiplies the fp32 scores); V's codes exactly with
 * their scale carried by the probabilities (block_size >= 32), or as code x the scale rounded
 * once to f16 (block_size 16), times a power of two per sequence and KV head that keeps the
 * values inside f16's range; q is converted to f16 exactly (a power of two per row), the
 * probabilities are f16 and fp32 accumulates.  Against the exact definition over code x scale
 * the output is then within half a bf16 ulp plus about 2^-11 of the largest |V| the row
 * attends to.
 * Supported: head_dim 64 or 128; n_q_heads / n_kv_heads a power of two <= 128;
 * B * n_kv_heads * ceil(max_q_len * n_q_heads / n_kv_heads / 256) < 2^31; scale positive and
 * finite.  Otherwise PKV_ERR_INVALID_ARG (nothing launched).  A chunk longer than its
 * context or a context longer than max_blocks*block_size is skipped and a block id outside the
 * pool is read as zeros; both are flagged (PKV_ERR_BOUNDS via pkv_check_device_error).  Every
 * wait in the kernel is bounded (2 s); on expiry the results are invalid and
 * pkv_check_device_error returns PKV_ERR_TIMEOUT.  No workspace; the caller owns every buffer. */
pkv_status pkv_prefill_attention(pkv_pool* pool, const void* q_dev, const int32_t* cu_q_lens_dev, int32_t max_q_len,
                                 const int32_t* block_tables_dev, int32_t max_blocks, const int32_t* context_lens_dev,
                                 int32_t B, int32_t n_q_heads, float scale, void* out_dev, pkv_stream_t stream);

/* pkv_append of the chunks' K/V (k_new/v_new [n_new][n_kv_heads][head_dim], slot_mapping
 * [n_new]) followed by pkv_prefill_attention, the attention launched as a programmatic
 * dependent of the append (as in pkv_decode_step).  Every argument is checked before anything
 * is launched. */
pkv_status pkv_prefill_step(pkv_pool* pool, const void* k_new_dev, const void* v_new_dev,
                            const int64_t* slot_mapping_dev, int64_t n_new, const void* q_dev,
                            const int32_t* cu_q_lens_dev, int32_t max_q_len, const int32_t* block_tables_dev,
                            int32_t max_blocks, const int32_t* context_lens_dev, int32_t B, int32_t n_q_heads,
                            float scale, void* out_dev, pkv_stream_t stream);

/* ------------------------------------------------------------------ decode attention without allocation
 * The pages have no counterpart to this call; it exists for callers that cannot allocate
 * device memory for a workspace: a plugin inside an engine that has already reserved nearly
 * all free device memory for its own KV pool (the serving stacks the pages describe hand
 * 85-92% of free memory to the KV cache), or a latency-critical decode loop that must not
 * call cudaMalloc because it can synchronise the device.
 *
 * Same computation, arguments and errors as pkv_decode_attention, minus the workspace: the
 * scratch is a fixed PKV_STATIC_WORKSPACE_BYTES array compiled into the library, which every
 * GPU that loads the library holds until the process exits.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine); it clears the merge tickets with
 * cudaMemsetAsync on `stream` and launches the same kernel.
 *   - Returns PKV_ERR_INVALID_ARG without launching when pkv_decode_workspace_bytes() for
 *     these B, n_q_heads, max_blocks exceeds PKV_STATIC_WORKSPACE_BYTES.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with the pool's device current; make that first call before any stream capture.
 *   - All calls share the one array, so calls that overlap on the GPU (other streams, other
 *     threads) race and corrupt each other's results: serialise them.
 *   - The looked-up address is kept for the life of the process.  cudaDeviceReset (or anything
 *     else that destroys the device's primary context) invalidates it: do not use this call on
 *     a device after resetting it. */
#define PKV_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)
pkv_status pkv_decode_attention_static(const pkv_pool* pool, const void* q_dev, const int32_t* block_tables_dev,
                                       int max_blocks, const int32_t* context_lens_dev, int B, int n_q_heads,
                                       float scale, void* out_dev, pkv_stream_t stream);

/* ------------------------------------------------------------------ host-driven steps
 * Kernel-driven copy for the per-step transfers of a decode step driven from the host (the
 * step's q/K/V, block tables, slots and lengths staged in pinned host memory, the output read
 * back): the SMs move 16-byte vectors instead of a copy engine, whose start-up dominates
 * transfers of this size.  The launch overhead of a decode step is what "TensorRT-LLM 推理加速
 * 实战" §7.1 removes with CUDA graphs; this copy can be captured into the same graph.
 *   dst, src: device memory of the current device, or host memory pinned with CUDA
 *             (cudaHostAlloc / cudaHostRegister), reached through its mapped address; both
 *             16-byte aligned, the ranges [p, p + bytes) must not overlap.
 *   bytes:    a multiple of 16; 0 is a no-op.
 * The caller owns both buffers and guarantees `bytes` lies inside each (as for a memcpy).
 * Asynchronous on `stream`; the host sees copied-to-host bytes after synchronising it.
 * PKV_ERR_INVALID_ARG (nothing launched): null or misaligned pointers, bytes % 16, overlap,
 * pageable host memory or another device's memory; PKV_ERR_CUDA: the launch failed. */
pkv_status pkv_stage_copy(void* dst, const void* src, size_t bytes, pkv_stream_t stream);

/* ------------------------------------------------------------------ testing and tuning
 * The library reads these environment variables when it loads, not on every call:
 *   PKV_TEST_WAIT_LIMIT_MS (> 0: every bounded wait in the kernels gives up after this many ms
 *   instead of 2 s), PKV_TEST_STALL_COPIES (non-zero: every pipeline stage waits for 16 bytes
 *   that no copy delivers, so the waits run out and calls report PKV_ERR_TIMEOUT: failure
 *   detection tested without a fault), PKV_ATTN_CTAS_PER_SM and PKV_ATTN_MAX_STAGES (decode
 *   attention launch shape; 0 or unset: the defaults).  Leave them unset in normal use.
 * pkv_debug_reload_env reads them again (for tests that switch the hooks on and off); it must
 * not run concurrently with other calls of the library. */
pkv_status pkv_debug_reload_env(void);

/* ------------------------------------------------------------------ utilities
 * KV memory ("TensorRT-LLM 推理加速实战" §8.1; aiqz.cc page, KV缓存管理):
 *   M_kv = 2 * n_layers * n_kv_heads * head_dim * n_tokens * batch * bytes_per_elem. */
uint64_t pkv_kv_bytes(int64_t n_layers, int64_t n_kv_heads, int64_t head_dim, int64_t n_tokens, int64_t batch,
                      double bytes_per_elem);

const char* pkv_status_str(pkv_status s);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
