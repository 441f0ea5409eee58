/*
 * pkv.h -- C ABI of libpkv.so: paged KV-cache writes and paged decode
 * attention on one GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes.  Device pointers point to
 * global memory of the current CUDA device; the caller owns every buffer
 * (the library never allocates or frees device memory).  All calls that
 * take a stream are asynchronous on that stream and return as soon as the
 * work is enqueued, except pkv_get_device_error, which synchronises it.
 *
 * Layouts (row-major, contiguous):
 *   q, out           [num_seqs, num_q_heads, head_dim]
 *   k, v (new)       [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache [num_blocks, num_kv_heads, block_size, head_dim]
 *                    one (block, kv head) tile is block_size * head_dim
 *                    contiguous elements
 *   block_tables     int32 [num_seqs, max_blocks_per_seq]
 *   seq_lens         int32 [num_seqs]
 *   slot_mapping     int64 [num_tokens], slot = block_id * block_size + offset
 *
 * Query head qh reads kv head qh / (num_q_heads / num_kv_heads).
 *
 * Error behaviour, common to all calls:
 *   - invalid arguments (null pointers, unsupported sizes or types,
 *     misaligned buffers) are rejected on the host before anything is
 *     enqueued: the call returns PKV_ERR_INVALID_ARG or PKV_ERR_UNSUPPORTED;
 *   - bad data met on the device (a block id outside the pool, a slot outside
 *     the cache, a sequence longer than its table) is never dereferenced: the
 *     element is skipped and a bit is set in a per-device error word, read
 *     and cleared by pkv_get_device_error;
 *   - a failed kernel launch returns PKV_ERR_CUDA.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,
  PKV_ERR_UNSUPPORTED = 2,
  PKV_ERR_CUDA = 3,
  PKV_ERR_WORKSPACE = 4
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Device error word bits. */
#define PKV_DEVERR_BAD_BLOCK_ID 0x1u   /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_BAD_SLOT 0x2u       /* slot >= num_blocks * block_size */
#define PKV_DEVERR_BAD_SEQ_LEN 0x4u    /* seq_len < 0 or beyond the table / hint */
#define PKV_DEVERR_WAIT_TIMEOUT 0x8u   /* a bounded wait on an async copy gave up */
#define PKV_DEVERR_SMEM_ALIGN 0x10u    /* shared memory not 1024-byte aligned for the swizzled
                                          tiles: the decode kernel returned without work */

/* Geometry and element type of one layer's K cache (the V cache is the same).
 * Supported: head_dim in {64, 128}; block_size in {8, 16, 32}; dtype any of
 * pkv_dtype. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  pkv_dtype dtype;
} pkv_cache_desc;

/*
 * pkv_kv_reshape_and_cache -- write each new token's K and V into its slot.
 *
 * "PagedAttention por dentro" (section "La tabla de páginas (block table)"):
 * a sequence's new token goes to the free position of its last block, or to
 * position 0 of a freshly appended block.  The host picks the slot; this call
 * performs the write: for every token t with slot_mapping[t] >= 0 and every
 * kv head h,
 *   k_cache[slot / bs][h][slot % bs][:] = convert(k[t][h][:])   (same for v)
 * convert is a copy (same type), an exact widening (bf16 -> f32), binary32 ->
 * bf16 round-to-nearest-even, or, for an fp8 cache, e4m3(x / kv_scale) with
 * the division in binary32, round-to-nearest-even and saturation to +-448.
 *
 *   k, v        device, [num_tokens, num_kv_heads, head_dim] of src_dtype
 *               (PKV_F32 or PKV_BF16), 16-byte aligned
 *   num_tokens  >= 0 (0 enqueues nothing)
 *   k_cache, v_cache, cache  destination caches, 16-byte aligned
 *   slot_mapping device int64 [num_tokens]; negative = skip the token;
 *               >= num_blocks * block_size sets PKV_DEVERR_BAD_SLOT and skips
 *   kv_scale    > 0, used only for fp8 caches
 * Two tokens with the same slot in one call race (the pages' allocator never
 * hands one slot to two tokens).
 */
pkv_status pkv_kv_reshape_and_cache(const void* k, const void* v, pkv_dtype src_dtype,
                                    int32_t num_tokens, void* k_cache, void* v_cache,
                                    const pkv_cache_desc* cache, const int64_t* slot_mapping,
                                    float kv_scale, pkv_stream_t stream);

/*
 * pkv_decode_workspace_bytes -- device workspace needed by
 * pkv_paged_attention_decode for this problem on the current device.
 *
 * Layout, both modes: a counter region of max(1 MiB, num_seqs * units * 4
 * bytes rounded up to 256) holding one merge counter per (sequence, kv-head
 * unit), then the mode's partials.  partition_tokens = 0 (balanced split):
 * the partial results of segments cut between thread blocks, two slots per
 * thread block of the largest grid; independent of the lengths.  partition_tokens > 0 (fixed
 * partitions): fp32 partials [num_seqs, num_q_heads, P, head_dim] and
 * [num_seqs, num_q_heads, P] maxima and sums, P = ceil(max_seq_len /
 * partition_tokens).  Returns 0 for invalid arguments.
 */
size_t pkv_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len,
                                  int32_t partition_tokens);

/*
 * pkv_paged_attention_decode -- one decode step of attention over paged K/V.
 *
 * For every sequence s and query head qh (kv head h = qh / g, g = Hq / Hkv):
 *   out[s][qh] = softmax_t(scale * q[s][qh] . K_s[t]) . V_s[t],  t < seq_lens[s]
 * where K_s[t] = k_cache[block_tables[s][t / bs]][h][t % bs] (and V alike):
 * the decode attention of "Optimización de Inferencia LLM" (section "El
 * Cuello de Botella de Atención del que Nadie Habla") read through the block
 * table as in "La despensa por casilleros" (section "El mecanismo: bloques,
 * block table y el gather del kernel"), with grouped-query sharing as in
 * "KV cache: la memoria de trabajo" (section "Trucos para que el cuaderno sea
 * más fino").  seq_lens counts the current token, whose K/V must already be
 * in the cache.  fp8 caches are read as code * kv_scale.  Accumulation is
 * binary32; out is rounded once (round-to-nearest-even) to q's type.  A
 * sequence with seq_len 0 gets a zero row.
 *
 *   out, q      device, [num_seqs, num_q_heads, head_dim] of q_dtype:
 *               PKV_F32 for an f32 cache, PKV_BF16 for bf16 and fp8 caches;
 *               16-byte aligned
 *   num_q_heads a multiple of cache->num_kv_heads
 *   block_tables, max_blocks_per_seq  device int32 table; entries past
 *               ceil(seq_len / bs) are never read
 *   seq_lens    device int32 [num_seqs]
 *   max_seq_len host upper bound of seq_lens (sizes the fixed-partition grid;
 *               a longer sequence sets PKV_DEVERR_BAD_SEQ_LEN and is clipped)
 *   partition_tokens  0 = balanced split over all SMs: the tiles of all
 *               (sequence, kv head) segments cut into equal ranges, one per
 *               warp; a segment cut between warps is merged by log-sum-exp
 *               in a second grid launched as the decode grid's programmatic
 *               dependent (tensor cores: two launches), or inside the decode
 *               grid by its last warp to finish (CUDA cores: one launch);
 *               > 0 = fixed KV partitions of that many tokens (a multiple
 *               of block_size), merged by pkv_split_kv_reduce inside this
 *               call (two launches)
 *   workspace   device, >= pkv_decode_workspace_bytes(...) bytes, 256-byte
 *               aligned.  Zero-fill it once before its first use; after that
 *               it serves any sequence of calls of either mode (and of
 *               pkv_cascade_decode and pkv_paged_attention_multi): every
 *               completed call leaves the merge counters of the first 1 MiB
 *               zero and no call writes partials there, and a balanced call
 *               whose counter region is larger (num_seqs * units > 262144)
 *               clears that region itself (an asynchronous memset on
 *               `stream`, before the decode) because an earlier call may
 *               have left partials in it.  Calls sharing one workspace must
 *               not overlap on the GPU.
 */
pkv_status pkv_paged_attention_decode(void* out, const void* q, pkv_dtype q_dtype,
                                      int32_t num_seqs, int32_t num_q_heads, const void* k_cache,
                                      const void* v_cache, const pkv_cache_desc* cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len, float scale,
                                      float kv_scale, int32_t partition_tokens, void* workspace,
                                      size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_paged_attention_decode_noalloc -- pkv_paged_attention_decode
 * (balanced split) for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart: this is a library convenience.
 * Some callers cannot supply the workspace the balanced split needs -- a
 * plugin inside a runtime that has reserved all device memory for its own
 * pool, plain C code that only receives tensor pointers, or a loop that must
 * not touch an allocator.  This call computes exactly what
 * pkv_paged_attention_decode computes with partition_tokens = 0, but keeps
 * its merge counters and partial results in a fixed 16 MiB scratch array in
 * device global memory that the library reserves on every GPU that loads it,
 * until the process exits.  It allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * Arguments are those of pkv_paged_attention_decode without
 * partition_tokens, workspace and workspace_bytes; layouts, supported shapes
 * and error behaviour are the same.  When the partial-result slots of a full
 * grid do not fit beside the merge counters, the call runs on fewer thread
 * blocks (same result).  A problem whose counters alone leave no room for
 * one thread block's slots (about four million (sequence, kv-head unit)
 * segments) is refused with PKV_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on a device looks up the scratch array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture.  Every call shares the one scratch array and clears
 * its counters at the start (an asynchronous memset on `stream`): calls that
 * overlap on the GPU -- on different streams, or from different threads --
 * race on it and must be serialised by the caller.
 */
pkv_status pkv_paged_attention_decode_noalloc(void* out, const void* q, pkv_dtype q_dtype,
                                              int32_t num_seqs, int32_t num_q_heads,
                                              const void* k_cache, const void* v_cache,
                                              const pkv_cache_desc* cache,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                              int32_t max_seq_len, float scale, float kv_scale,
                                              pkv_stream_t stream);

/*
 * pkv_paged_attention_decode_window -- pkv_paged_attention_decode over a
 * sliding window with attention sinks: a sequence of length L > window_tokens
 * attends only its first sink_tokens tokens and its last window_tokens tokens
 * ("PagedAttention por dentro", sections "Sliding window attention" and
 * "StreamingLLM (Xiao et al., 2024): los attention sinks").  The blocks that
 * hold no attended token are never read, nor their table entries (an engine
 * frees the blocks that fell out of the window; the entries may hold
 * anything).  A sequence with L <= window_tokens attends every token.
 *
 *   window_tokens  > 0; 0 makes the call pkv_paged_attention_decode
 *   sink_tokens    >= 0, ignored without a window
 *
 * Every other argument, the workspace (the same size as
 * pkv_decode_workspace_bytes gives) and the error behaviour are those of
 * pkv_paged_attention_decode; negative window_tokens or sink_tokens give
 * PKV_ERR_INVALID_ARG.
 */
pkv_status pkv_paged_attention_decode_window(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs,
                                             int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                             const pkv_cache_desc* cache, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                             int32_t max_seq_len, float scale, float kv_scale, int32_t window_tokens,
                                             int32_t sink_tokens, int32_t partition_tokens, void* workspace,
                                             size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_cascade_workspace_bytes -- bytes of device workspace pkv_cascade_decode
 * needs for this problem (0 for invalid sizes, a batch too large for the
 * counter region described below, or no current device): the workspace of a
 * balanced pkv_paged_attention_decode call, then the prefix partial result
 * (num_seqs * num_q_heads rows of head_dim + 4 fp32 values: the unnormalised
 * output, the running maximum, the running sum, two of padding), then one
 * such partial per piece the prefix pass may cut the prefix into (the pieces
 * fill one wave of the GPU; at most 32).
 */
size_t pkv_cascade_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t max_seq_len);

/*
 * pkv_cascade_decode -- pkv_paged_attention_decode for a batch whose block
 * tables all begin with the same prefix_blocks physical blocks (requests
 * that share a system prompt: "PagedAttention por dentro", section "Prefix
 * caching cross-session"; "La despensa por casilleros", section "Prefix
 * caching: compartir casilleros con copy-on-write").  The result is the one
 * pkv_paged_attention_decode gives on the same arguments; only the order of
 * the work differs:
 *
 *   1. one kernel attends every query row of the batch (num_seqs * group rows
 *      per kv head) over the shared prefix blocks, so each prefix block is
 *      read once per call instead of once per sequence, and leaves a partial
 *      result per row (unnormalised output, running maximum, running sum) in
 *      the workspace;
 *   2. the decode kernel attends each sequence over its own blocks after the
 *      prefix, starting each sequence's online softmax from the prefix
 *      partial (the log-sum-exp algebra of split-KV decoding).
 *
 * A sequence shorter than the prefix attends only its first seq_lens[i]
 * tokens of it, as in plain decoding.
 *
 *   prefix_blocks  number of leading table entries every sequence shares,
 *                  0 <= prefix_blocks <= max_blocks_per_seq; 0 makes the call
 *                  a plain pkv_paged_attention_decode.  The prefix blocks are
 *                  read through the first sequence's table, which must hold
 *                  all prefix_blocks entries; every other sequence's entries
 *                  for the prefix blocks it attends are compared with the
 *                  first's, and a differing entry raises
 *                  PKV_DEVERR_BAD_BLOCK_ID
 *   workspace      at least pkv_cascade_workspace_bytes(...) bytes of device
 *                  memory, 256-byte aligned, owned by the caller.  Its first
 *                  1 MiB holds merge counters, as for
 *                  pkv_paged_attention_decode: the decode's at the bottom,
 *                  the prefix pass's (num_kv_heads * ceil(num_seqs * group /
 *                  16) of them) at the top.  They must be zero when a call
 *                  starts and every completed call leaves them zero, so a
 *                  workspace zero-filled once serves any sequence of decode
 *                  and cascade calls.  A batch whose two counter sets do not
 *                  fit in 1 MiB gets PKV_ERR_UNSUPPORTED
 *
 * Every other argument is that of pkv_paged_attention_decode (the
 * partitioning is always the balanced one).  Caches of PKV_F32 give
 * PKV_ERR_UNSUPPORTED: the prefix pass runs on the tensor cores, which take
 * bf16 and fp8 operands.  All arguments are validated before anything is
 * enqueued; errors as for pkv_paged_attention_decode.
 */
pkv_status pkv_cascade_decode(void* out, const void* q, pkv_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                              const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t max_seq_len, int32_t prefix_blocks, float scale, float kv_scale,
                              void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_multi_workspace_bytes -- bytes of device workspace
 * pkv_paged_attention_multi needs (0 for invalid sizes, a batch too large for
 * the counter region below, or no current device): the 1 MiB counter region,
 * then, when the K/V range is cut into pieces, one partial row of head_dim + 4
 * fp32 values per query row, query head and piece (at most 32 pieces); for
 * calls the multi-query decode serves (pkv_multi_kernel_for), at least its
 * balanced split's partial slots (16 rows each, two per thread block).
 *   max_q   the largest number of query tokens of one sequence
 */
size_t pkv_multi_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim);

/*
 * pkv_paged_attention_multi -- paged attention for several query tokens per
 * sequence: a chunk of a chunked prefill, or the tokens a speculative step
 * verifies ("PagedAttention por dentro", section "Chunked prefill integrado
 * con paged KV"; "Componentes Internos de Servicio de vLLM", section
 * "Chunked prefill protege la cola del TTFT").  The chunk's K and V are
 * already in the cache (pkv_kv_reshape_and_cache first, as in decode).
 *
 *   out[r][qh] = softmax_t(scale * q[r][qh] . K_s[t]) . V_s[t]
 *                over t = 0 .. seq_lens[s] - T + i
 *
 * for the i-th of the T = q_start[s+1] - q_start[s] query rows of sequence s,
 * r = q_start[s] + i: the chunk is the sequence's last T positions and each
 * of its tokens attends every position up to its own (causal inside the
 * chunk).  T = 1 for every sequence is decode.  The query heads of a kv head
 * are grouped as in pkv_paged_attention_decode.
 *
 *   out, q        device [total_q, num_q_heads, head_dim], bf16 (q_dtype
 *                 PKV_BF16), 16-byte aligned; out is written only
 *   q_start       device int32 [num_seqs + 1], q_start[0] = 0, non-decreasing,
 *                 q_start[num_seqs] = total_q
 *   max_q         host upper bound of T (sizes the grid); T > max_q, T >
 *                 seq_lens[s] or a row past total_q sets PKV_DEVERR_BAD_SEQ_LEN
 *                 and leaves the sequence's rows unwritten
 *   caches        bf16 or fp8-e4m3 (PKV_F32 gives PKV_ERR_UNSUPPORTED: the
 *                 products run on the tensor cores); block tables, seq_lens,
 *                 max_seq_len, scale and kv_scale as for
 *                 pkv_paged_attention_decode
 *   workspace     >= pkv_multi_workspace_bytes(...) bytes of device memory,
 *                 256-byte aligned, its first 1 MiB zero when the call starts
 *                 (every completed call leaves it zero; the same region as
 *                 the decode's counters)
 *
 * All arguments are validated before anything is enqueued; errors as for
 * pkv_paged_attention_decode.
 */
pkv_status pkv_paged_attention_multi(void* out, const void* q, pkv_dtype q_dtype, const int32_t* q_start,
                                     int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_q_heads,
                                     const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* seq_lens, int32_t max_seq_len, float scale, float kv_scale,
                                     void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * pkv_multi_kernel_for -- the kernel pkv_paged_attention_multi launches for a
 * call of this shape under the current pkv_set_tcgen05 setting.  Host only:
 * nothing is enqueued and no device is needed.  The three kernels compute the
 * same attention; they differ in how the rows are tiled.
 *
 *   PKV_MULTI_TCGEN05       128-row tiles on the tcgen05 tensor cores: a
 *                           (sequence, kv head) with max_q * Hq / Hkv >= 128,
 *                           or a cache shape the mma.sync kernel has no
 *                           instance of
 *   PKV_MULTI_QUERY_DECODE  the balanced decode kernel with 16 (token, head)
 *                           rows per unit, each row limited to the positions
 *                           up to its token: max_q * Hq / Hkv <= 32, Hq / Hkv
 *                           a power of two up to 16, and an instance for the
 *                           cache (bf16: head_dim 128 with blocks of 8, 16 or
 *                           32, head_dim 64 with 16; fp8-e4m3: blocks of 16);
 *                           with its merge grid, two launches
 *   PKV_MULTI_MMA_SYNC      16-row tiles on mma.sync (every other call)
 *   PKV_MULTI_NONE          the shape is invalid (num_seqs < 0, max_q <= 0, a
 *                           bad cache descriptor, Hq not a multiple of Hkv)
 *                           or no kernel serves it (PKV_ERR_UNSUPPORTED)
 */
typedef enum {
  PKV_MULTI_NONE = 0,
  PKV_MULTI_TCGEN05 = 1,
  PKV_MULTI_QUERY_DECODE = 2,
  PKV_MULTI_MMA_SYNC = 3
} pkv_multi_kernel;

pkv_multi_kernel pkv_multi_kernel_for(int32_t num_seqs, int32_t max_q, int32_t num_q_heads,
                                      const pkv_cache_desc* cache);

/*
 * pkv_decode_step -- one decode step of one layer: pkv_kv_reshape_and_cache of
 * the step's new tokens, then pkv_paged_attention_decode, on `stream`.
 *
 * This is the iteration of "vLLM en Kubernetes" (section "Continuous
 * batching: dejar de esperar al más lento": every step produces one token
 * per live session) restricted to
 * one attention layer: the new tokens' K/V enter the cache ("PagedAttention
 * por dentro", section "La tabla de páginas (block table)"), then each
 * sequence attends over all its cached tokens.  The result is identical to the
 * two calls made one after the other.  The decode grid is launched as a
 * programmatic dependent of the cache-write grid: it reads lengths, block
 * tables and q while the cache write runs, and waits for the write to finish
 * before it reads any K/V.  So q, out, block_tables and seq_lens must not be
 * produced by the cache write, which is always the case here.  (The merge
 * grid of a balanced split on the tensor cores follows the decode grid as
 * in pkv_paged_attention_decode.)
 *
 * Arguments: those of pkv_kv_reshape_and_cache (k, v, src_dtype,
 * num_new_tokens, slot_mapping, caches, kv_scale) and of
 * pkv_paged_attention_decode (the rest).  All arguments are validated before
 * anything is enqueued.
 */
pkv_status pkv_decode_step(const void* k, const void* v, pkv_dtype src_dtype, int32_t num_new_tokens,
                           const int64_t* slot_mapping, void* k_cache, void* v_cache,
                           const pkv_cache_desc* cache, void* out, const void* q, pkv_dtype q_dtype,
                           int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t max_seq_len, float scale, float kv_scale,
                           int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                           pkv_stream_t stream);

/*
 * pkv_split_kv_reduce -- log-sum-exp merge of per-partition partial results.
 *
 * The pages do not describe a split of the KV sequence; this is the algebra
 * of a softmax over disjoint token sets.  For each (s, qh), over the first
 * n = ceil(seq_lens[s] / partition_tokens) partitions:
 *   M = max_p m_part[p];  w_p = l_part[p] * exp(m_part[p] - M);
 *   out = sum_p w_p * o_part[p] / sum_p w_p          (zero row when n = 0)
 *
 *   o_part  device fp32 [num_seqs, num_q_heads, max_partitions, head_dim],
 *           each partition's output already normalised by its own sum
 *   m_part  device fp32 [num_seqs, num_q_heads, max_partitions]: the largest
 *           scaled score scale * q . k of the partition (natural-log units)
 *   l_part  device fp32 [...]: sum over the partition of exp(score - m)
 *   out     device [num_seqs, num_q_heads, head_dim] of out_dtype (F32/BF16)
 */
pkv_status pkv_split_kv_reduce(void* out, pkv_dtype out_dtype, const float* o_part,
                               const float* m_part, const float* l_part, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                               int32_t partition_tokens, int32_t max_partitions,
                               pkv_stream_t stream);

/*
 * pkv_gather_kv -- contiguous copy of every sequence's cached tokens (test
 * and export aid): k_out[cu_seq_lens[s] + t][h][:] =
 * k_cache[block_tables[s][t / bs]][h][t % bs][:] for t < seq_lens[s], byte
 * for byte ("La despensa por casilleros", section "El mecanismo: bloques,
 * block table y el gather del kernel": the blocks read as if contiguous).
 *
 *   k_out, v_out  device [sum(seq_lens), num_kv_heads, head_dim] of the
 *                 cache's type
 *   cu_seq_lens   device int64 [num_seqs + 1], exclusive prefix of seq_lens
 *   max_seq_len   host upper bound of seq_lens (sizes the grid)
 */
pkv_status pkv_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                         const pkv_cache_desc* cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                         const int64_t* cu_seq_lens, int32_t num_seqs, int32_t max_seq_len,
                         pkv_stream_t stream);

/*
 * pkv_copy_blocks -- copy whole blocks (K and V, every kv head) from one
 * block pool to another, or within one pool.
 *
 * Two uses in the pages: copy-on-write, where sequences that share a
 * physical block diverge and the branch about to write gets its own copy
 * first ("PagedAttention por dentro", section "Copy-on-write para sampling
 * paralelo"; "La despensa por casilleros", section "Prefix caching:
 * compartir casilleros con copy-on-write"); and swap, where a preempted
 * sequence's blocks move to host memory and later come back ("PagedAttention
 * por dentro", section "Evicción y preemption: qué hace cuando el pool se
 * agota", the swap strategy).
 *
 *   k_dst, v_dst  destination pool [dst->num_blocks, Hkv, bs, d]
 *   k_src, v_src  source pool [src->num_blocks, Hkv, bs, d]: same block_size,
 *                 num_kv_heads, head_dim and dtype as the destination (the
 *                 pools may differ in num_blocks)
 *   block_pairs   int64 [num_pairs][2], (source block, destination block)
 *
 * Every pointer is a device address: device memory, or page-locked host
 * memory mapped into the device's address space (as cudaHostAlloc returns
 * it), which is how a swap reaches host memory.  The pools are 16-byte
 * aligned, block_pairs 8-byte aligned.  The copies of one call run
 * concurrently: a destination block must not be the source or the
 * destination of another pair of the same call.  The copy is bit-exact.  A
 * pair with an id outside its pool sets PKV_DEVERR_BAD_BLOCK_ID and is
 * skipped.  Asynchronous on `stream`.
 */
pkv_status pkv_copy_blocks(void* k_dst, void* v_dst, const pkv_cache_desc* dst, const void* k_src,
                           const void* v_src, const pkv_cache_desc* src, const int64_t* block_pairs,
                           int32_t num_pairs, pkv_stream_t stream);

/*
 * pkv_get_device_error -- synchronise `stream`, then read and clear the
 * current device's error word (PKV_DEVERR_* bits) into *code_out.
 */
pkv_status pkv_get_device_error(uint32_t* code_out, pkv_stream_t stream);

/*
 * pkv_selftest_wait_timeout -- exercise the failure path of the bounded
 * waits (no counterpart on the source pages: a diagnostic of this library).
 *
 * Every kernel that waits for an asynchronous copy waits with an iteration
 * limit of about a second, after which it sets PKV_DEVERR_WAIT_TIMEOUT,
 * stops issuing copies and returns, so that a lost copy cannot hang the
 * GPU.  This call launches one thread that arms an mbarrier for 16 bytes of
 * transactions no copy will deliver (it issues none, so nothing is left in
 * flight) and waits on it with that same bounded wait: the wait gives up,
 * the bit is set in the device error word and the kernel returns, leaving
 * the context usable.  Takes up to about a second of GPU time.
 * Asynchronous on `stream`; read the bit with pkv_get_device_error.
 */
pkv_status pkv_selftest_wait_timeout(pkv_stream_t stream);

/* Human-readable name of a status; never NULL. */
const char* pkv_status_string(pkv_status status);

/* Number of SMs of the current device, or 0 on error (the balanced split
 * sizes its grid from it). */
int32_t pkv_device_sm_count(void);

/*
 * Which units run the two contractions of the decode (q.K and P.V) for bf16
 * and fp8 caches.  The softmax, its online rescaling and every accumulation
 * stay in fp32 either way ("Optimización de Inferencia LLM", section
 * "PagedAttention: Conceptos de SO se Encuentran con Memoria GPU"); fp32
 * caches always use the CUDA cores.
 *
 *   PKV_ENGINE_TENSOR_CORES (default)  the G query heads of a kv head are the
 *       rows of an m16n8k16 MMA against each K and V tile, fp32 accumulate;
 *       probabilities enter P.V as a head plus a remainder of the operand
 *       type (~16 significant bits).  Fewer instructions per KV byte: the
 *       decode stays bound by HBM at 8 query heads per kv head and for fp8.
 *   PKV_ENGINE_CUDA_CORES  every product is a packed fp32 FMA on the CUDA
 *       cores (probabilities in fp32).
 *
 * Process-wide; applies to decode calls issued after it returns (calls in
 * flight keep the engine they were issued with).  PKV_ERR_INVALID_ARG for an
 * unknown value.
 */
typedef enum { PKV_ENGINE_TENSOR_CORES = 0, PKV_ENGINE_CUDA_CORES = 1 } pkv_decode_engine;

pkv_status pkv_set_decode_engine(pkv_decode_engine engine);
pkv_decode_engine pkv_get_decode_engine(void);

/*
 * The tcgen05 kernels of pkv_paged_attention_multi and of the prefix pass of
 * pkv_cascade_decode (bf16 caches, and fp8-e4m3 caches with head_dim 128).
 *
 *   enable != 0 (default)  a call whose tiles can hold 128 query rows -- a
 *       (sequence, kv head) with max_q * Hq / Hkv >= 128, or a cascade batch
 *       with num_seqs * Hq / Hkv >= 128 -- runs the tcgen05 kernel: 128 rows
 *       per CTA, q.K and P.V as 5th-generation tensor-core MMAs with both
 *       accumulators in tensor memory, K/V tiles by tensor copy (fp8 codes
 *       widened exactly to fp16 in shared memory). Smaller calls keep the
 *       mma.sync kernels, except for cache shapes those have no instance of
 *       (fp8 caches with 8- or 32-token blocks), which the tcgen05 kernel
 *       serves at any size.
 *   enable == 0            every call runs the mma.sync kernels (fp8 caches
 *       with 8- or 32-token blocks are then PKV_ERR_UNSUPPORTED).
 *
 * Both give the same results within the tolerances of their cache type; the
 * switch exists to compare them. Process-wide, for calls issued after it
 * returns.
 */
void pkv_set_tcgen05(int32_t enable);
int32_t pkv_get_tcgen05(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
