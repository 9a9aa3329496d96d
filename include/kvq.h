/*
 * kvq.h -- C ABI of the paged quantized KV-cache library (GB300, sm_103a).
 *
 * One decode step of an LLM over a block-paged KV cache held in INT8 / FP8
 * codes with fp32 scales (or plain FP16 for selected layers):
 *
 *   kvq_alloc_pool   one pool of fixed-size physical blocks per layer
 *   kvq_append       quantize the new tokens' K/V and scatter them into slots
 *   kvq_paged_decode attention of each new Q over its sequence's cached K/V,
 *                    reached through a block table, dequantized on the fly
 *
 * Sources (the pages this method is described on):
 *   [KVC]  "KV Cache优化实战：大模型推理显存占用与加速方案详解",
 *          0539edu.com/news/5800990
 *   [P402] xpshop.cn/articles/article-402.html (INT8 KV + paged cache)
 *   [P312] xpshop.cn/articles/article-312.html (PagedAttention + FP8/INT8 KV)
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers unless a comment says "host".
 *   - fp16 data is IEEE binary16, passed as kvq_half (its 16 bits).
 *   - Every call that takes a stream is asynchronous on that stream; its
 *     return value reports only the host-side argument checks (and launch
 *     errors).  Errors found on the device -- a slot or block id outside the
 *     pool, a context longer than the caller promised, a pipeline wait that
 *     ran out -- set an error word inside the pool; the offending token or
 *     block is skipped and nothing faults.  kvq_get_error() reads and clears it.
 *     While the error word reports OUT_OF_RANGE or TIMEOUT for a decode, the
 *     contents of that decode's `out` are undefined (rows of a skipped block
 *     or of a warp that gave up may be partial, zero or left as they were).
 *   - The library allocates device memory only in kvq_alloc_pool (and only when
 *     the caller passes no buffer).  Decode scratch ("workspace") comes from
 *     the caller.
 *   - Thread safety: calls on different pools may run concurrently; calls on
 *     one pool must be ordered by the caller (one stream, or events).
 *   - One-time set-up the library remembers (kernel shared-memory opt-ins, the
 *     address of kvq_paged_decode_noalloc's array) is kept per CUDA context,
 *     keyed on the context current on the calling thread: after
 *     cudaDeviceReset, or in another driver context, it is done again.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvq_half; /* IEEE binary16 bits */

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent shape      */
    KVQ_ERR_UNSUPPORTED = 2,  /* valid but not built (head_dim, group, block)    */
    KVQ_ERR_CUDA = 3,         /* a CUDA runtime call failed                      */
    KVQ_ERR_OUT_OF_RANGE = 4, /* device: slot / block id / length out of range   */
    KVQ_ERR_WORKSPACE = 5,    /* decode workspace smaller than required          */
    KVQ_ERR_TIMEOUT = 6       /* device: a bounded pipeline wait gave up         */
} kvq_status;

/* Cache formats ([KVC] §2.3: INT8 absmax-symmetric with per-token, per-channel
 * or per-group scales; FP8; [KVC] §3.3 / [P312] §三: selected layers stay FP16). */
typedef enum {
    KVQ_FP16 = 0,              /* fp16 values, no scale                              */
    KVQ_INT8_PER_TOKEN = 1,    /* one fp32 scale per (token, K|V) over all kv heads  */
    KVQ_INT8_PER_CHANNEL = 2,  /* static fp32 scale per (K|V, kv head, channel)      */
    KVQ_INT8_PER_GROUP = 3,    /* one fp32 scale per `group` contiguous channels of
                                  one (token, kv head, K|V) vector                   */
    KVQ_FP8_E4M3_PER_TOKEN = 4, /* e4m3 codes, one fp32 scale per (token, K|V)       */
    KVQ_INT4_PER_GROUP = 5,    /* 4-bit codes in [-7, 7] ([KVC] §2.3 lists INT4 beside
                                  INT8/FP8), scale = absmax/7 per `group` channels as
                                  for KVQ_INT8_PER_GROUP; two codes per byte         */
    KVQ_FP8_E5M2 = 6           /* e5m2 codes of the values themselves, no scale
                                  ([P312] §三: kv_cache_dtype fp8_e5m2); saturating  */
} kvq_dtype;

typedef struct kvq_pool kvq_pool; /* opaque; one per layer */

/* Byte accounting of a pool ([KVC] §1.2: KV bytes = 2 x tokens x kv_heads x
 * head_dim x bytes per layer).  code_bytes is exactly that formula for
 * num_blocks*block_size tokens; scales and the small header are separate. */
typedef struct {
    size_t total_bytes;  /* everything kvq_alloc_pool needs (header + regions)  */
    size_t code_bytes;   /* 2 * num_blocks * block_size * kv_heads * head_dim * elem */
    size_t scale_bytes;  /* fp32 scales of every format that has them           */
    size_t header_bytes; /* device error word and padding                       */
    size_t page_bytes;   /* bytes of one (block, kv head) page: K+V codes (+ group scales) */
} kvq_pool_layout;

/* Byte accounting for the given geometry, without allocating.  Returns
 * KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED for a geometry kvq_alloc_pool would
 * refuse.  `out` is a host pointer.  Host only; needs no GPU. */
kvq_status kvq_pool_layout_query(int64_t num_blocks, int block_size, int kv_heads,
                                 int head_dim, kvq_dtype dtype, int group,
                                 kvq_pool_layout* out);

/* Total bytes of kvq_pool_layout_query (0 for a refused geometry). */
size_t kvq_pool_bytes(int64_t num_blocks, int block_size, int kv_heads, int head_dim,
                      kvq_dtype dtype, int group);

/* Create a pool ([KVC] §2.2 PagedAttention: fixed-size physical blocks, e.g.
 * 16 tokens, reached through a per-request block table; [P312] §三: blocks of
 * 16 or 32 tokens).
 *   num_blocks : physical blocks (>= 1)
 *   block_size : tokens per block: 8, 16, 32 or 64 ([KVC] §3.2: 8 for short
 *                contexts at high concurrency, 16 or 32 for long ones); other
 *                sizes return UNSUPPORTED.  INT4 pools take 16 or more; pools
 *                of 8-token blocks serve append, decode and block copy, while
 *                kvq_prefill and the cascade with prefix_blocks > 0 refuse
 *                them with UNSUPPORTED.
 *   kv_heads   : KV heads (>= 1); head_dim: 64 or 128
 *   group      : channels per scale for KVQ_INT8_PER_GROUP / KVQ_INT4_PER_GROUP
 *                (a multiple of 16 that divides head_dim); ignored otherwise
 *   device_buf : caller-owned device memory of buf_bytes >= kvq_pool_bytes(..),
 *                256-byte aligned; NULL makes the library cudaMalloc (and later
 *                cudaFree) the pool on the current device.
 *   out        : host pointer that receives the handle.
 * The pool's contents are unspecified until written by kvq_append, except
 * that the error word is cleared and per-channel scales are set to zero.
 * Synchronous.  Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
kvq_status kvq_alloc_pool(int64_t num_blocks, int block_size, int kv_heads, int head_dim,
                          kvq_dtype dtype, int group, void* device_buf, size_t buf_bytes,
                          kvq_pool** out);

/* Release the handle; frees device memory only if the library allocated it.
 * Synchronises the device first when it frees.  NULL is accepted. */
kvq_status kvq_free_pool(kvq_pool* pool);

/* KVQ_INT8_PER_CHANNEL only: set the static scales ([KVC] §2.3 "per-channel:
 * a scale per channel").  k_scale, v_scale: fp32 [kv_heads][head_dim] device
 * arrays, copied into the pool on `stream`.  A zero scale quantizes its
 * channel to code 0. */
kvq_status kvq_set_channel_scales(kvq_pool* pool, const float* k_scale, const float* v_scale,
                                  cudaStream_t stream);

/* KVQ_INT8_PER_CHANNEL only: calibrate the static scales from T tokens:
 * scale[kv][h][d] = max_t |x[t][h][d]| / 127 (fp32).  k, v: [T][kv_heads][head_dim]
 * fp16.  T >= 1. */
kvq_status kvq_calibrate_channel_scales(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                                        int64_t T, cudaStream_t stream);

/* Quantize and scatter T new tokens ([KVC] §1.1: the decode step appends the
 * new token's K/V to the cache; §2.3: absmax symmetric quantization).
 *   k, v         : fp16 [T][kv_heads][head_dim]
 *   slot_mapping : int64 [T]; token i goes to block slot/block_size, offset
 *                  slot%block_size.  A negative slot skips the token.
 * Per format: scale s = absmax/127 (INT8 dynamic), absmax/7 (INT4) or
 * absmax/448 (FP8 e4m3), fp32 IEEE division; code = clamp(round_half_even(x/s),
 * -127, 127) for INT8 (-7, 7 for INT4), e5m2 round-to-nearest-even of x
 * itself saturating at 57344 for KVQ_FP8_E5M2,
 * e4m3 round-to-nearest-even saturating for FP8; an all-zero group stores s=0
 * and zero codes.  Per-channel uses the pool's static scales.  FP16 stores x.
 * Two tokens with the same slot in one call race (result unspecified).
 * Device errors: a slot >= num_blocks*block_size sets OUT_OF_RANGE and the
 * token is skipped. */
kvq_status kvq_append(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                      const int64_t* slot_mapping, int64_t T, cudaStream_t stream);

/* Copy whole blocks ([KVC] §4.4: a request that must write into a block it
 * shares with others first gets its own copy -- copy-on-write).
 *   src_blocks, dst_blocks : int32 [n]; block dst_blocks[i] becomes a copy of
 *                            block src_blocks[i]: every kv head's K and V codes,
 *                            their per-group scales, and (per-token formats)
 *                            the block's token scales
 * Pairs run in parallel: a destination must not be another pair's source or
 * destination.  Device errors: an id outside the pool sets OUT_OF_RANGE and
 * that pair is skipped. */
kvq_status kvq_copy_blocks(kvq_pool* pool, const int32_t* src_blocks, const int32_t* dst_blocks,
                           int n, cudaStream_t stream);

/* Per-head mixed precision ([P312] §六: the attention heads that quantization
 * hurts stay FP16, the others are quantized): hold two pools per layer over a
 * contiguous split of the kv heads (permute the heads once so that the FP16
 * ones come first) and address each pool's slice of the full per-token rows
 * with a row stride.
 *   kvq_append_strided      : kvq_append with k, v pointing at the pool's first
 *                             kv head; token t's K/V row starts row_stride
 *                             elements after token t-1's (row_stride >=
 *                             kv_heads*head_dim, a multiple of 8)
 *   kvq_paged_decode_strided: kvq_paged_decode with q pointing at the first Q
 *                             head of the pool's groups and sequence s's row
 *                             q_row_stride elements after s-1's (a multiple of
 *                             8, >= num_q_heads*head_dim); out likewise with
 *                             out_row_stride (>= num_q_heads*head_dim), so the
 *                             two pools' calls fill disjoint heads of one
 *                             output.  num_q_heads counts this pool's Q heads. */
kvq_status kvq_append_strided(kvq_pool* pool, const kvq_half* k, const kvq_half* v,
                              int64_t row_stride, const int64_t* slot_mapping, int64_t T,
                              cudaStream_t stream);
kvq_status kvq_paged_decode_strided(const kvq_pool* pool, const kvq_half* q,
                                    int64_t q_row_stride, int num_seqs, int num_q_heads,
                                    const int32_t* block_table, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context_len,
                                    float sm_scale, float* out, int64_t out_row_stride,
                                    void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes kvq_paged_decode needs for these sizes (split-K partials).
 * May be 0.  Host only. */
size_t kvq_decode_workspace_bytes(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                  int max_context_len);

/* Decode attention over the paged cache ([KVC] §1.1 decode step, §2.1 GQA,
 * §2.2 block table, §2.3 quantized KV; §4.3: dequantization fused into the
 * attention kernel rather than a separate pass).
 *   q             : fp16 [num_seqs][num_q_heads][head_dim]; num_q_heads is a
 *                   multiple of kv_heads; Q head hq reads kv head hq / (num_q_heads/kv_heads)
 *   block_table   : int32 [num_seqs][max_blocks_per_seq] physical block ids
 *   context_lens  : int32 [num_seqs] tokens to attend (after this step's append)
 *   max_context_len : host-side upper bound of context_lens, <= max_blocks_per_seq*block_size
 *   sm_scale      : softmax scale (usually 1/sqrt(head_dim))
 *   out           : fp32 [num_seqs][num_q_heads][head_dim]
 *   workspace     : >= kvq_decode_workspace_bytes(..) bytes, 256-byte aligned
 *                   (may be NULL when that is 0)
 * out = softmax(q . k^T * sm_scale) v over tokens 0..L-1, with k^, v^ = code * scale.
 * A sequence with L == 0 gets zeros.  Device errors: a block id outside the
 * pool sets OUT_OF_RANGE and that block is skipped; L > max_context_len sets
 * OUT_OF_RANGE and L is clamped.  Host errors beyond the argument checks:
 * UNSUPPORTED when num_seqs > 65535 or when two shared-memory stages of one
 * (block, kv head) page for each of a CTA's 4 warps exceed 227 KB (FP16
 * pages of 64-token blocks at head_dim 128); the workspace query then
 * returns 0. */
kvq_status kvq_paged_decode(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                            int num_q_heads, const int32_t* block_table,
                            int max_blocks_per_seq, const int32_t* context_lens,
                            int max_context_len, float sm_scale, float* out,
                            void* workspace, size_t ws_bytes, cudaStream_t stream);

/* As kvq_paged_decode, with an explicit split of each sequence's blocks across
 * thread blocks: split_blocks > 0 forces that many blocks per split (split-K
 * over the context, merged by log-sum-exp); 0 picks automatically. */
size_t kvq_decode_workspace_bytes_ex(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                     int max_context_len, int split_blocks);
kvq_status kvq_paged_decode_ex(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                               int num_q_heads, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* context_lens,
                               int max_context_len, float sm_scale, float* out,
                               void* workspace, size_t ws_bytes, int split_blocks,
                               cudaStream_t stream);

/* One whole decode step of one layer ([KVC] §1.1: the new token's K/V joins
 * the cache, then the new Q attends over everything cached, itself included):
 * kvq_append of one token per sequence followed by kvq_paged_decode.
 *   k_new, v_new : fp16 [num_seqs][kv_heads][head_dim], 16-byte aligned;
 *                  sequence s's token is stored at position context_lens[s]-1,
 *                  i.e. in block block_table[s][(L-1)/block_size], offset
 *                  (L-1)%block_size (the caller has already counted it in L
 *                  and mapped its block)
 *   the other arguments and the result are those of kvq_paged_decode, with
 *   workspace sized by kvq_decode_workspace_bytes.
 * Results equal kvq_append (slots derived as above) then kvq_paged_decode on
 * the same stream.  A sequence with L == 0 stores nothing; L > max_context_len
 * stores nothing and sets OUT_OF_RANGE (the decode clamps as documented); a
 * negative block id at position L-1 sets OUT_OF_RANGE and stores nothing.
 * The append starts once everything before it on the stream has completed,
 * and the decode is launched as its programmatic dependent: the decode's
 * set-up and its first page fetches overlap the append, and the one page per
 * sequence that the append writes (the block holding position L-1) is read
 * only after the append is done.  So the block receiving a sequence's new
 * token must be read by no other sequence except as that sequence's own last
 * block (a block shared further must be copied first, kvq_copy_blocks);
 * otherwise the other sequence may see the block before or after the write.
 * The caller's k_new/v_new/q buffers must stay valid until the stream reaches
 * this call, as for every other call. */
kvq_status kvq_decode_step(kvq_pool* pool, const kvq_half* k_new, const kvq_half* v_new,
                           const kvq_half* q, int num_seqs, int num_q_heads,
                           const int32_t* block_table, int max_blocks_per_seq,
                           const int32_t* context_lens, int max_context_len, float sm_scale,
                           float* out, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Shared-prefix ("cascade") decode ([KVC] §2.2, §4.4: requests with a common
 * prefix -- a system prompt, a fixed history -- share its physical blocks): the first
 * prefix_blocks blocks of every sequence are the same physical blocks, those
 * of block_table row 0.  They are read once per kv head for all sequences'
 * Q heads (a partial softmax per (sequence, Q head)), the remaining blocks by
 * the paged decode, and the two parts are combined by log-sum-exp.
 *   prefix_blocks : 0 <= prefix_blocks <= max_blocks_per_seq; 0 is plain
 *                   kvq_paged_decode
 *   workspace     : >= kvq_cascade_workspace_bytes(..) bytes, 256-byte aligned
 *   the other arguments and the result are those of kvq_paged_decode.
 * Precondition (not checked): block_table[s][j] == block_table[0][j] for
 * every j < prefix_blocks and every s whose context reaches block j.
 * Sequences shorter than the prefix are handled (their rows stop at their own
 * length).  Results equal kvq_paged_decode's up to fp32 rounding order.
 * Pools of 8-token blocks: prefix_blocks > 0 returns UNSUPPORTED. */
size_t kvq_cascade_workspace_bytes(const kvq_pool* pool, int num_seqs, int num_q_heads,
                                   int max_context_len);
kvq_status kvq_cascade_decode(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                              int num_q_heads, const int32_t* block_table,
                              int max_blocks_per_seq, const int32_t* context_lens,
                              int max_context_len, int prefix_blocks, float sm_scale,
                              float* out, void* workspace, size_t ws_bytes,
                              cudaStream_t stream);

/* Prefill / chunked prefill ([KVC] §1.1: the prompt's tokens are processed
 * together, each attending causally to every token up to itself; a long prompt
 * may be split into chunks, each attending to the cache the earlier chunks
 * wrote): attention of each sequence's new query tokens over its paged cache.
 *   q             : fp16 [Tq][num_q_heads][head_dim], Tq = q_start[num_seqs]
 *   q_start       : int32 [num_seqs + 1] (device); sequence s's query tokens
 *                   are rows q_start[s] .. q_start[s+1]-1, n_s of them
 *   max_q_len     : host-side upper bound of n_s (sizes the grid)
 *   context_lens  : int32 [num_seqs]: L_s tokens in the cache, this chunk's
 *                   included -- its K/V must already be appended (kvq_append);
 *                   query token i sits at position L_s - n_s + i
 *   out           : fp32 [Tq][num_q_heads][head_dim]
 * out[row] = softmax(q . k^T * sm_scale) v over positions 0 .. L_s - n_s + i.
 * Device errors: L_s < n_s or L_s > max_context_len sets OUT_OF_RANGE (L_s is
 * clamped; rows with no position left get zeros); a block id outside the
 * pool sets OUT_OF_RANGE and that block is skipped.  No workspace.  Pools of
 * 8-token blocks return UNSUPPORTED. */
kvq_status kvq_prefill(const kvq_pool* pool, const kvq_half* q, int num_seqs, int num_q_heads,
                       const int32_t* q_start, int max_q_len, const int32_t* block_table,
                       int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                       float sm_scale, float* out, cudaStream_t stream);

/* kvq_prefill in two passes through a caller workspace (same arguments and
 * results, [KVC] §1.1).  Every 64-token key step of a sequence's cache is
 * read by all the thread blocks whose query rows come after it; here a first
 * pass turns each step's codes into exact fp16 once, with its per-token scales
 * beside them, and the attention pass reads those instead of converting the
 * codes again in every block.  The arithmetic is the same as kvq_prefill's
 * (codes exact in fp16, scales applied outside the contraction).
 *   workspace : >= kvq_prefill_workspace_bytes(pool, num_seqs, max_context_len)
 *               bytes, 256-byte aligned, owned by the caller; its contents are
 *               scratch (written and read by this call only)
 * kvq_prefill_workspace_bytes returns 0 for the formats this path does not take
 * (per-group formats with more than one group per head, 8-token blocks); for
 * them kvq_prefill_ex ignores the workspace and runs kvq_prefill.  Returns
 * KVQ_ERR_WORKSPACE when the workspace is missing or too small. */
size_t kvq_prefill_workspace_bytes(const kvq_pool* pool, int num_seqs, int max_context_len);
kvq_status kvq_prefill_ex(const kvq_pool* pool, const kvq_half* q, int num_seqs, int num_q_heads,
                          const int32_t* q_start, int max_q_len, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* context_lens,
                          int max_context_len, float sm_scale, float* out, void* workspace,
                          size_t ws_bytes, cudaStream_t stream);

/* kvq_decode_step with the cascade decode: the new token of sequence s goes to
 * position context_lens[s]-1, which must lie past the shared prefix (a token
 * written into a shared block would change every sequence's prefix). */
kvq_status kvq_cascade_decode_step(kvq_pool* pool, const kvq_half* k_new, const kvq_half* v_new,
                                   const kvq_half* q, int num_seqs, int num_q_heads,
                                   const int32_t* block_table, int max_blocks_per_seq,
                                   const int32_t* context_lens, int max_context_len,
                                   int prefix_blocks, float sm_scale, float* out,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Maximum split-K scratch of kvq_paged_decode_noalloc, in bytes (16 MiB). */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)

/* kvq_paged_decode_ex for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for library users.
 * Some callers must not allocate: a serving loop whose memory is all reserved
 * up front, code running under a custom or capped allocator that refuses new
 * requests, or host code in a context where a cudaMalloc would stall or is
 * not permitted.  This call takes no workspace: the split-K scratch lives in
 * a fixed array of KVQ_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library keeps until the process exits.  Arguments and
 * results are those of kvq_paged_decode_ex; the caller still provides q,
 * the table, the lengths and `out`.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call in a CUDA context looks up that device's copy of the
 *     array (cudaGetSymbolAddress, with the context current), so make that
 *     first call before any stream capture; later calls in the same context
 *     reuse the address, and a new context (after cudaDeviceReset, say) gets a
 *     fresh lookup on its first call.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose execution
 *     overlaps on the GPU -- on two streams, or from two threads -- race on
 *     it; order them.
 *   - Returns KVQ_ERR_WORKSPACE, launching nothing, when the scratch the call
 *     needs (kvq_decode_workspace_bytes_ex for the same sizes) exceeds
 *     KVQ_NOALLOC_SCRATCH_BYTES; KVQ_ERR_CUDA if the array cannot be located. */
kvq_status kvq_paged_decode_noalloc(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                                    int num_q_heads, const int32_t* block_table,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    int max_context_len, float sm_scale, float* out,
                                    int split_blocks, cudaStream_t stream);

/* Self-test of the bounded pipeline waits (the pages have no counterpart):
 * kvq_paged_decode with sm_scale 1, except that the first page copy of the
 * grid's first warp is announced to its barrier but never issued, so that
 * wait cannot complete.  Every wait of the call gives up after wait_tries
 * tries of at most ~1 ms (1 <= wait_tries <= 1000); the warp then sets
 * KVQ_ERR_TIMEOUT in the pool's error word, waits (bounded the same way) for
 * its other copies in flight and exits.  Nothing hangs or faults and the
 * context stays usable; kvq_get_error() then returns KVQ_ERR_TIMEOUT.  The
 * outputs of the units that warp held are unspecified.  Arguments as for
 * kvq_paged_decode. */
kvq_status kvq_selftest_decode_timeout(const kvq_pool* pool, const kvq_half* q, int num_seqs,
                                       int num_q_heads, const int32_t* block_table,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int max_context_len, float* out, void* workspace,
                                       size_t ws_bytes, int wait_tries, cudaStream_t stream);

/* Read back n slots in a canonical layout (for tests and debugging).
 *   codes_out  : [n][2][kv_heads][head_dim] elements of the pool's code type
 *                (int8, e4m3 byte, or fp16; INT4 codes come back one per int8)
 *   scales_out : per-group [n][2][kv_heads][head_dim/group] fp32;
 *                per-token [n][2] fp32; may be NULL (and is ignored) for
 *                FP16 and per-channel pools
 * A slot outside the pool sets OUT_OF_RANGE and its output is left untouched. */
kvq_status kvq_read_slots(const kvq_pool* pool, const int64_t* slots, int64_t n,
                          void* codes_out, float* scales_out, cudaStream_t stream);

/* Synchronise `stream`, read and clear the pool's device error word.
 * Returns KVQ_OK, KVQ_ERR_OUT_OF_RANGE or KVQ_ERR_TIMEOUT (the first that is set). */
kvq_status kvq_get_error(kvq_pool* pool, cudaStream_t stream);

/* Static description of a status code (never NULL). */
const char* kvq_status_string(kvq_status status);

/* Per-kernel timing (a measurement aid; no result depends on it).  A library
 * call may run several kernels (kvq_paged_decode: the decode kernel, then the
 * split merge; kvq_decode_step: the append, the decode, the merge;
 * kvq_prefill_ex: the staging kernel, then the attention kernel).  This call
 * hands the calling host thread's next n kernel launches one event each:
 * right after the library launches its k-th kernel from now (k = 0 .. n-1,
 * counted across calls, on this thread only), it records events[k] on that
 * kernel's stream.  With an event of the caller's own recorded just before
 * the call, the differences time each kernel on the device.  A launch that
 * would follow a recorded event as a programmatic dependent just waits for it
 * instead (no overlap), so timed kernels run one after another.  After n
 * launches nothing more is recorded; a new call replaces what is left, and
 * n = 0 (events may then be NULL) clears it.
 *   events : host array of n CUDA events (cudaEvent_t), created and owned by
 *            the caller; copied, so the array may be reused after the call
 *   n      : 0 .. KVQ_MAX_PHASE_EVENTS
 * Returns KVQ_ERR_INVALID_ARG for n outside that range or NULL events with
 * n > 0.  A record that fails (an event of another device, say) makes the
 * launching call return KVQ_ERR_CUDA without launching that call's later
 * kernels, so its results are then undefined. */
#define KVQ_MAX_PHASE_EVENTS 8
kvq_status kvq_set_phase_events(const cudaEvent_t* events, int n);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
