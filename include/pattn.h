/*
 * pattn.h -- C ABI of the GB300 (sm_103a) paged variable-length attention
 * library, libpattn.so.
 *
 * One call computes exact softmax attention for a batch of requests that
 * mixes prefills, chunked prefills and single-token decodes, over a paged KV
 * cache.  The operation is defined on these pages:
 *   - "[vLLM] FlashAttention", FlashAttentionBackend.get_kv_cache_shape:
 *     the cache is (2, num_blocks, block_size, num_kv_heads, head_size), index
 *     0 of the first dimension is K and 1 is V, and block_size must be a
 *     multiple of 16;
 *   - same page, FlashAttentionImpl.__init__: num_queries_per_kv =
 *     num_heads / num_kv_heads query heads share one KV head (GQA);
 *   - same page, FlashAttentionMetadata: query_start_loc, seq_lens,
 *     block_table, max_query_len, max_seq_len let one call serve requests of
 *     different lengths;
 *   - "[vLLM] other attention backends", TritonAttentionMetadata:
 *     seq_len = context_len + query_len, so query row i of a request sits at
 *     position context_len + i;
 *   - "RBLN Attention modes", overview / Full Attention / SWA: scores over the
 *     valid tokens, softmax, product with V; causal masking; a sliding window;
 *     per-partition results merged with online softmax;
 *   - "[vLLM] FlashAttention", "why this design" item 4: tiled online softmax
 *     is exact attention, not an approximation.
 *
 * For request r: q_len = query_start_loc[r+1] - query_start_loc[r],
 * s = seq_lens[r], ctx = s - q_len.  Row i (position p = ctx + i) of head h
 * reads KV head g = h / (num_heads / num_kv_heads).  Key k < s lives in
 * physical block block_table[r * max_blocks_per_seq + k / block_size], slot
 * k % block_size.  Key k is visible iff (causal == 0 or k <= p) and
 * (window <= 0 or p - k < window).  out = softmax(scale * q . K^T over the
 * visible keys) . V.  A request with q_len == 1 is a decode (the page
 * "[vLLM] Lightning & Linear Attention", prefill/decode split with
 * threshold 1); any other q_len > 0 is a prefill; q_len == 0 produces nothing.
 *
 * Conventions for every entry point
 *   - Device pointers are marked [device]; everything else is host memory.
 *   - The caller owns every buffer.  The library allocates no memory, keeps
 *     no state between calls and may be called from several host threads.
 *   - Work is enqueued on ext->stream and the call returns without waiting.
 *   - Errors are returned, never thrown, and no call aborts the process.
 */
#ifndef PATTN_H
#define PATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PATTN_OK = 0,
  PATTN_ERR_INVALID_ARGUMENT = 1,   /* NULL pointer, bad size, bad scale     */
  PATTN_ERR_UNSUPPORTED = 2,        /* valid but not built (head_size, ...)  */
  PATTN_ERR_WORKSPACE_TOO_SMALL = 3,
  PATTN_ERR_CUDA = 4,               /* a CUDA runtime call failed            */
  PATTN_ERR_BAD_METADATA = 5,       /* device-detected: see read_device_status */
  PATTN_ERR_DEVICE_TIMEOUT = 6      /* device-detected: a bounded wait expired */
} pattn_status_t;

typedef enum {
  PATTN_KV_BF16 = 0,      /* K and V stored as bf16                          */
  PATTN_KV_FP8_E4M3 = 1,  /* K and V stored as e4m3 bytes, one fp32 scale each */
  PATTN_KV_F16 = 2        /* K and V stored as f16; q and out are f16 too (the
                             FlashAttention backend supports float16 and
                             bfloat16 models)                                 */
} pattn_kv_dtype_t;

/*
 * Host-side sizes and resources of one call.  Everything a device-pointer API
 * cannot learn without a device-to-host copy is passed here, so no call ever
 * synchronises.  The FlashAttentionMetadata fields (num_actual_tokens,
 * max_query_len, max_seq_len) have the same meaning.
 */
typedef struct {
  size_t struct_size;     /* sizeof(pattn_ext_t)                              */
  int num_seqs;           /* B: requests in the batch                         */
  int num_tokens;         /* T: rows of q and out (>= query_start_loc[B])     */
  int max_blocks_per_seq; /* row stride of block_table                        */
  int num_blocks;         /* physical blocks in kv_cache                      */
  int max_query_len;      /* >= every q_len in the batch                      */
  int max_seq_len;        /* >= every seq_len in the batch                    */
  int num_splits;         /* decode KV partitions: 0 = library chooses,
                             1..PATTN_MAX_SPLITS forces the count             */
  void* workspace;        /* [device] scratch of >= workspace_bytes, 256-B aligned */
  size_t workspace_bytes;
  void* stream;           /* cudaStream_t; NULL = the legacy default stream   */
  void* const* timing_events; /* optional host array of 8 cudaEvent_t, or NULL.
                             If set, events [2k] and [2k+1] are recorded on
                             stream right before and after phase k: 0 plan,
                             1 prefill, 2 decode, 3 combine (a phase that does
                             not run records both back to back).  For
                             profiling; the caller owns the events.          */
  const float* sinks;     /* [device] fp32 [num_heads] attention-sink logits, or
                             NULL for none.  Head h's sink joins the softmax
                             normaliser as a term with no value:
                               out = sum_k e^{s_k} V_k / (e^{sinks[h]} + sum_k e^{s_k}),
                             s_k = scale * q . k (the sink is not scaled).  A
                             sink of -inf is no sink; values must be finite or
                             -inf.  The pages ("RBLN Attention modes", Full
                             Attention: flash attention serves layers with
                             attention sinks) give no formula; this is the
                             reading taken.  A caller built against the
                             header without this field passes the smaller
                             struct_size and gets no sinks.                  */
  int head_size_v;        /* 0: K and V share head_size and the cache is
                             [2, num_blocks, block_size, num_kv_heads, head_size].
                             > 0: the DiffKV layout ("[vLLM] other attention
                             backends", FlashAttention DiffKV: V has its own
                             head size and the cache is asymmetric; the page
                             gives no shape, this is the reading taken): the
                             cache is [num_blocks, block_size, num_kv_heads,
                             head_size + head_size_v], each row the token's K
                             then its V, and out is [num_tokens, num_heads,
                             head_size_v].  head_size and head_size_v are then
                             multiples of 32 up to 256, the cache is bf16 or
                             f16 (PATTN_KV_F16), and a generic (not tensor-core)
                             kernel serves every row.  A caller built against
                             the header without this field gets 0.           */
} pattn_ext_t;

#define PATTN_MAX_SPLITS 64

/*
 * pattn_varlen_fwd -- the forward pass.
 *
 *   q               [device] bf16 [num_tokens, num_heads, head_size], contiguous
 *                   (f16 when kv_dtype is PATTN_KV_F16)
 *   kv_cache        [device] [2, num_blocks, block_size, num_kv_heads, head_size],
 *                   contiguous, bf16 or e4m3 bytes per kv_dtype; 16-B aligned
 *   block_table     [device] int32 [num_seqs, max_blocks_per_seq]; entries past
 *                   ceil(seq_len / block_size) are never read
 *   seq_lens        [device] int32 [num_seqs]
 *   query_start_loc [device] int32 [num_seqs + 1], non-decreasing prefix sum
 *   out             [device] bf16 (f16 with PATTN_KV_F16) [num_tokens, num_heads,
 *                   head_size]; rows of
 *                   tokens outside [query_start_loc[0], query_start_loc[B]) are
 *                   left untouched
 *   scale           multiplies q . k; finite and >= 0
 *   num_heads, num_kv_heads   num_heads % num_kv_heads == 0 and
 *                   num_heads / num_kv_heads <= 16
 *   head_size       64 or 128 (with ext->head_size_v > 0: the K head size, a
 *                   multiple of 32 up to 256; see pattn_ext_t.head_size_v)
 *   block_size      a multiple of 16 (the ValueError of get_kv_cache_shape)
 *   window          <= 0: no window; > 0: keys with p - k < window are visible
 *   causal          1: k <= p; 0: every key < seq_len (then window must be <= 0)
 *   kv_dtype        a pattn_kv_dtype_t.  With e4m3, decode rows run on the
 *                   bandwidth-bound decode kernel and prefill rows on the
 *                   tensor-core prefill kernel.  At head_size 128 its score
 *                   MMAs take the K codes as they are, against each q row
 *                   split exactly into two e4m3 codes per value after a
 *                   power-of-two scaling, and V tiles are widened to f16
 *                   (exactly) for f16 P V MMAs; at 64 K and V are widened and
 *                   q is scaled per row into f16 (the decode kernel likewise
 *                   per head)
 *   kv_scale        host float[2] {k_scale, v_scale}; required for e4m3, ignored
 *                   for bf16 (may be NULL)
 *   ext             host sizes, workspace and stream (see pattn_ext_t)
 *
 * Returns PATTN_OK once the work is enqueued.  Host-side checks return
 * INVALID_ARGUMENT / UNSUPPORTED / WORKSPACE_TOO_SMALL before any CUDA call;
 * a failed launch returns PATTN_ERR_CUDA.  Metadata the host cannot see
 * (q_len > seq_len, a block id outside [0, num_blocks), seq_len above
 * max_blocks_per_seq * block_size or max_seq_len) is detected on the device:
 * the offending ids are clamped so no access leaves the buffers, the rows of
 * that request are unspecified but finite, and a status word in the
 * workspace records it for pattn_read_device_status.
 */
pattn_status_t pattn_varlen_fwd(const void* q, const void* kv_cache,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const int32_t* query_start_loc, void* out, float scale,
                                int num_heads, int num_kv_heads, int head_size,
                                int block_size, int window, int causal, int kv_dtype,
                                const float* kv_scale, const pattn_ext_t* ext);

/*
 * Workspace bytes pattn_varlen_fwd needs for these sizes (reads num_seqs,
 * num_tokens, max_query_len, max_seq_len and num_splits from ext; ignores its
 * workspace and stream).  Returns 0 if the arguments are invalid.
 */
size_t pattn_workspace_bytes(const pattn_ext_t* ext, int num_heads, int num_kv_heads,
                             int head_size, int block_size);

/*
 * The decode KV partition count pattn_varlen_fwd will use for these sizes
 * (ext->num_splits if set, else the library's choice).  Partitions are runs of
 * ceil(n / splits) whole KV blocks over the n blocks a decode row can see,
 * merged by log-sum-exp ("RBLN Attention modes", flash attention; the Triton
 * backend's 16 parallel softmax segments).
 */
int pattn_decode_splits(const pattn_ext_t* ext, int num_heads, int num_kv_heads,
                        int block_size, int window);

/*
 * Reads and clears the device status word of ext->workspace.  Synchronises
 * ext->stream.  Returns PATTN_OK, PATTN_ERR_BAD_METADATA or
 * PATTN_ERR_DEVICE_TIMEOUT for the calls since the last read (each
 * pattn_varlen_fwd call first clears the word on its stream), or
 * PATTN_ERR_CUDA if the copy fails.
 */
pattn_status_t pattn_read_device_status(const pattn_ext_t* ext);

/*
 * pattn_decode_fwd_static -- the decode rows of a batch, with no workspace.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot allocate device memory or hand over a workspace: a plugin inside
 * an application whose allocator owns all device memory, or code on a
 * latency-critical path where cudaMalloc / cudaFree would synchronise the
 * device.  It computes exactly what pattn_varlen_fwd computes for the requests
 * with query_len == 1 (same kernels, same partition count for the same sizes),
 * leaves the rows of every other request untouched, and allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments are those of pattn_varlen_fwd; the sizes of pattn_ext_t are passed
 * directly and `stream` is a cudaStream_t (NULL = legacy default stream).
 * Scratch comes from a fixed device array of PATTN_STATIC_SCRATCH_BYTES
 * inside the library, held by every GPU that loads the library until the
 * process exits.  A batch whose partials need more
 * (num_seqs * num_heads * splits * (head_size + 1) * 4 bytes, roughly) returns
 * PATTN_ERR_WORKSPACE_TOO_SMALL before any GPU work; pass a smaller
 * num_splits or use pattn_varlen_fwd.  Every call looks up the array's device
 * address in the current context (cudaGetSymbolAddress, which allocates
 * nothing), so the device that owns `stream` must be current; the first call
 * in a context may load the library's device code, so make it before any
 * stream capture.  Any context the runtime API can make current is served
 * (the primary one, or one a host application created and made current).
 * All calls share the array and it keeps the last call's contents: the
 * status word and the partition counters are cleared on `stream` at the start
 * of each call; calls whose work may overlap on the GPU (different streams or
 * host threads) race and must be serialised by the caller.  Requests with
 * query_len != 1 are skipped: their output rows are neither read nor written
 * and they are not reported.  Device-detected metadata errors of the decode
 * rows (a block id outside the pool, seq_len beyond the block table) are
 * clamped as in pattn_varlen_fwd, those rows are zeroed, and nothing is
 * reported (there is no workspace to read a status from).
 */
#define PATTN_STATIC_SCRATCH_BYTES (32u << 20)
pattn_status_t pattn_decode_fwd_static(const void* q, const void* kv_cache,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       const int32_t* query_start_loc, void* out, float scale,
                                       int num_heads, int num_kv_heads, int head_size,
                                       int block_size, int window, int causal, int kv_dtype,
                                       const float* kv_scale, int num_seqs, int num_tokens,
                                       int max_blocks_per_seq, int num_blocks, int max_seq_len,
                                       int num_splits, void* stream);

/*
 * pattn_cascade_fwd -- pattn_varlen_fwd for a batch whose requests all start
 * with the same cached prefix ("[vLLM] FlashAttention", Cascade Attention;
 * FlashAttentionMetadata.use_cascade / common_prefix_len).
 *
 * The prefix's attention is computed once for every query token of the batch
 * (one request of num_tokens queries over common_prefix_len keys, not causal:
 * every query sits after the prefix), each request's suffix (its keys past
 * the prefix) separately and causally, and the two are merged by
 * log-sum-exp.  The result is pattn_varlen_fwd's up to rounding; the prefix's
 * K/V pages are read once for the batch instead of once per request.
 *
 * Arguments are pattn_varlen_fwd's, plus common_prefix_len: a positive
 * multiple of block_size, at most max_seq_len.  The first
 * common_prefix_len / block_size block-table entries of every request must
 * name the same blocks (the pass reads row 0's), and every request's cached
 * context (seq_len - query_len) must cover the prefix; a request whose
 * context does not is reported as bad metadata (its rows are finite but
 * unspecified).  causal must be 1 and window <= 0 (else
 * PATTN_ERR_UNSUPPORTED); bf16, f16 and e4m3 caches are served as by
 * pattn_varlen_fwd.  The workspace comes from
 * pattn_cascade_workspace_bytes: besides the two passes' own scratch it holds
 * their fp32 partial results, 2 * num_tokens * num_heads * (head_size + 1)
 * floats.  The status word is read with pattn_read_device_status as usual.
 */
pattn_status_t pattn_cascade_fwd(const void* q, const void* kv_cache,
                                 const int32_t* block_table, const int32_t* seq_lens,
                                 const int32_t* query_start_loc, void* out, float scale,
                                 int num_heads, int num_kv_heads, int head_size,
                                 int block_size, int window, int causal, int kv_dtype,
                                 const float* kv_scale, int common_prefix_len,
                                 const pattn_ext_t* ext);

/* Workspace bytes pattn_cascade_fwd needs (0 if the arguments are invalid). */
size_t pattn_cascade_workspace_bytes(const pattn_ext_t* ext, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int common_prefix_len);

/*
 * pattn_reshape_and_cache -- write new key and value rows into the paged cache.
 *
 * The step that fills the cache pattn_varlen_fwd reads ("[vLLM]
 * FlashAttention", FlashAttentionMetadata.slot_mapping; the cache-write
 * kernel of the DiffKV backend in "[vLLM] other attention backends").
 *
 *   key, value      [device] bf16 [num_tokens, num_kv_heads, head_size],
 *                   contiguous, 16-B aligned
 *   kv_cache        [device] the cache of pattn_varlen_fwd, 16-B aligned,
 *                   updated in place
 *   slot_mapping    [device] int64 [num_tokens]: token t goes to block
 *                   slot / block_size, offset slot % block_size; a negative
 *                   slot writes nothing (padding).  Slots of one call must be
 *                   distinct (two tokens on one slot leave either's row).
 *   head_size       a multiple of 8; block_size a multiple of 16
 *   kv_dtype        bf16: the bits are copied; e4m3: each element x is stored
 *                   as e4m3(x / scale) (fp32 division, round to nearest even,
 *                   saturated at +-448, NaN stays NaN), scale = kv_scale[0]
 *                   for K and kv_scale[1] for V (host floats, > 0, finite)
 *   device_status   [device] optional (may be NULL): a slot at or beyond
 *                   num_blocks * block_size writes nothing and ORs
 *                   PATTN_ERR_BAD_METADATA's device bit (1) into this word
 *   stream          a cudaStream_t (NULL = legacy default stream)
 *
 * Returns PATTN_OK once enqueued; argument errors before any CUDA call;
 * PATTN_ERR_CUDA if the launch fails.  Allocates nothing, never synchronises.
 */
pattn_status_t pattn_reshape_and_cache(const void* key, const void* value, void* kv_cache,
                                       const int64_t* slot_mapping, int num_tokens,
                                       int num_kv_heads, int head_size, int block_size,
                                       int num_blocks, int kv_dtype, const float* kv_scale,
                                       unsigned* device_status, void* stream);

/*
 * pattn_reshape_and_cache_diffkv -- pattn_reshape_and_cache for the DiffKV
 * layout (pattn_ext_t.head_size_v; the DiffKV backend of "[vLLM] other
 * attention backends" has its own cache-write kernel for its asymmetric
 * cache).
 *
 *   key             [device] 16-bit [num_tokens, num_kv_heads, head_size]
 *   value           [device] 16-bit [num_tokens, num_kv_heads, head_size_v]
 *   kv_cache        [device] [num_blocks, block_size, num_kv_heads,
 *                   head_size + head_size_v], updated in place: token t's key
 *                   row then its value row go to row [s / block_size]
 *                   [s % block_size][h], s = slot_mapping[t]
 *   head_size, head_size_v   multiples of 8; block_size a multiple of 16
 *   kv_dtype        PATTN_KV_BF16 or PATTN_KV_F16 (the bits are copied)
 *   slot_mapping, device_status, stream   as for pattn_reshape_and_cache
 *
 * All buffers 16-B aligned.  Returns PATTN_OK once enqueued; argument errors
 * before any CUDA call.  Allocates nothing, never synchronises.
 */
pattn_status_t pattn_reshape_and_cache_diffkv(const void* key, const void* value,
                                              void* kv_cache, const int64_t* slot_mapping,
                                              int num_tokens, int num_kv_heads, int head_size,
                                              int head_size_v, int block_size, int num_blocks,
                                              int kv_dtype, unsigned* device_status,
                                              void* stream);

/* A static, human-readable name for a status code. */
const char* pattn_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int pattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PATTN_H */
