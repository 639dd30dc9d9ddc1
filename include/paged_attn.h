/*
 * paged_attn.h - C ABI of the GB300 (sm_103a) paged KV attention library.
 *
 * FlashAttention-style attention over a block-paged KV cache with grouped-query
 * heads: a cache write, a split-KV decode (partials + log-sum-exp combine) and a
 * causal varlen kernel for prefill, speculative verify and mixed batches.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller. The library never
 *   allocates, frees or synchronises inside a call; work is enqueued on `stream`
 *   (a cudaStream_t passed as void*; NULL = the legacy default stream). Calls are
 *   therefore legal inside CUDA-graph capture.
 * - Layouts are dense row-major (last index fastest):
 *     q, out          [N, Hq, D]                 (N = sequences for decode, tokens for varlen)
 *     k_cache/v_cache [num_blocks, block_size, Hkv, D]
 *     block_tables    [R, max_blocks_per_seq] int32, a row's unused tail may hold any page id
 *     key/value       [num_tokens, Hkv, D]
 *   Every tensor pointer must be 16-byte aligned.
 * - dtype: PA_DTYPE_BF16 (bf16 storage, fp32 scores/softmax/accumulation, probabilities
 *   rounded to bf16 for the P.V product) or PA_DTYPE_F32 (fp32 throughout, no TF32).
 * - Positions come from device buffers (lengths, query_start_loc), never from launch
 *   arguments, so a captured graph stays valid as sequences grow. Launch shapes depend
 *   only on the host integers of each call.
 * - Shape and scalar errors are refused on the host before anything is enqueued.
 *   Data errors that only the device can see (a page id outside the pool, a length
 *   beyond the table, a slot outside the pool, a query block longer than its
 *   sequence) are clamped or skipped so that no kernel reads or writes out of bounds;
 *   if `error_word` is non-NULL (a device int32 the caller zeroes) the kernel ORs a
 *   PA_ERRBIT_* bit into it. No kernel traps or asserts.
 *
 * Sources of the operations (by page title and section):
 *   "32. Production attention kernels": One kernel for the whole batch (unified varlen
 *     kernel, GQA packing, positions from lengths); Long contexts: split the keys
 *     (split-KV partials, log-sum-exp merge, split-count heuristic); Quantized KV
 *     caches (write through slot_mapping).
 *   "TileInfer.jl - Attention kernels": Walking the block table; Decode: GQA packing and
 *     split-KV (unnormalised fp32 partials, neutral partials for empty splits).
 *   "poot - Attention and KV Cache": Split-KV decode ((o, m, l) partials, combine);
 *     KV cache (write map, -1 = padding token writes nothing).
 *   "paged-attn-xpu": Usage (paged_attention_decode argument list, scale default),
 *     Validation (empty context gives zeros).
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, Hq % Hkv != 0, misalignment */
  PA_ERR_UNSUPPORTED = 2,        /* a shape or dtype this build has no kernel for           */
  PA_ERR_WORKSPACE_TOO_SMALL = 3,
  PA_ERR_CUDA = 4                /* a CUDA runtime/driver call failed (launch, tensor map)  */
} pa_status;

typedef enum pa_dtype {
  PA_DTYPE_F32 = 0,
  PA_DTYPE_BF16 = 1,
  PA_DTYPE_INT8 = 2,      /* 8-bit cache codes (the *_quant calls only) */
  PA_DTYPE_FP8_E4M3 = 3   /* 8-bit cache codes (the *_quant calls only) */
} pa_dtype;

/* Bits a kernel ORs into *error_word (see conventions above). */
#define PA_ERRBIT_PAGE_OUT_OF_POOL   1  /* table entry outside [0, num_blocks): that page reads as zeros   */
#define PA_ERRBIT_LENGTH_OUT_OF_RANGE 2 /* length < 0 or > max_blocks_per_seq*block_size: decode clamps it,
                                           varlen zeroes that request's rows                            */
#define PA_ERRBIT_SLOT_OUT_OF_POOL   4  /* slot >= num_blocks*block_size or < -1: token not written         */
#define PA_ERRBIT_QUERY_LAYOUT       8  /* query_start_loc not monotone or q_len > seq_len: rows zeroed     */
#define PA_ERRBIT_WAIT_TIMEOUT      16  /* an internal bounded wait expired: that tile's output is invalid */

/* Optional score modifiers for the *_ex entry points (a NULL options pointer, or a
 * zero-initialised struct, means none of them).
 *   sliding_window > 0: a query at position t sees only keys at positions > t - sliding_window
 *     (and <= t when causal). "32. Production attention kernels", One kernel for the whole
 *     batch: the window's loop start and extra mask term.
 *   logit_softcap > 0: every score s = scale * q.k becomes logit_softcap * tanh(s / logit_softcap)
 *     before the softmax. "poot - Attention and KV Cache", The streaming schedule
 *     (softcap_or_identity) and Implementation details.
 *   sinks: NULL or a device pointer to Hq float32 sink logits (natural-log units): query head h's
 *     softmax denominator gains e^{sinks[h]} and no value is added, so
 *     out = sum_p e^{s_p} v_p / (e^{sinks[h]} + sum_p e^{s_p}). "32. Production attention
 *     kernels", Stretch exercises, item 4 (attention sinks). Must be 4-byte aligned. */
typedef struct pa_attn_options {
  int32_t sliding_window;
  float logit_softcap;
  const float* sinks;
} pa_attn_options;

/* Row strides for the *_strided entry points, in ELEMENTS of the tensor's dtype (a NULL pointer,
 * or 0 in a field, means dense rows of Hq * D elements).
 *   q:   elements from one query row to the next (a sequence for decode, a token for varlen),
 *        e.g. (Hq + 2 * Hkv) * D when q is the query slice of a fused QKV projection output;
 *   out: likewise for the output rows.
 * Within a row the Hq heads stay dense (D elements apart). A non-zero stride must be at least
 * Hq * D (rows never overlap) and a whole number of 16-byte units (a multiple of 8 elements for
 * bf16, 4 for f32), else PA_ERR_INVALID_ARGUMENT. The pages pass dense tensors; the strided form
 * takes the row layouts a serving engine's projections produce without a copy. */
typedef struct pa_row_strides {
  int64_t q;
  int64_t out;
} pa_row_strides;

/* Human-readable name of a status code. Never NULL. */
const char* pa_status_string(int status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int pa_version(void);

/* Supported-shape query: 1 if the decode (is_varlen=0) or varlen (is_varlen=1) entry point
 * has a kernel for this head_dim / group / block_size / dtype, else 0. Host only. */
int pa_supports(int is_varlen, int head_dim, int num_q_heads, int num_kv_heads,
                int block_size, pa_dtype dtype);

/* Split-count heuristic of the decode path (host only, no CUDA call).
 * Source: "32. Production attention kernels", Long contexts: split the keys (choose_splits:
 * enough programs to fill the GPU, no split smaller than a few blocks, at most 32), taken
 * further here: splits of at least `min_chunks_per_split` chunks are preferred (each CTA pays a
 * fixed start-up and merge cost), and among those the count whose CTAs best fill whole waves
 * of `num_sms * ctas_per_sm` resident CTAs; when such long splits leave less than one wave,
 * the count that fills one wave (splits of at least 4 chunks).
 *   num_units            = num_seqs * num_kv_heads (CTAs per split)
 *   max_chunks           = cdiv(max_blocks_per_seq * block_size, 16) (16-token chunks per row)
 *   min_chunks_per_split = preferred shortest split (the library uses 64 for bf16, 256 for
 *                          8-bit caches); values below 4 act as 4
 * Returns a count in [1, 32]; 1 for degenerate inputs. */
int pa_plan_decode_splits(int num_units, int max_chunks, int num_sms, int ctas_per_sm, int min_chunks_per_split);

/* The split count an auto (num_splits = 0) pa_paged_attention_decode call with these sizes
 * uses on the CURRENT device (queries the SM count and the kernel's occupancy once per
 * device). Returns 0 for arguments the decode call would refuse. */
int pa_decode_auto_splits(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int max_blocks_per_seq, pa_dtype dtype);

/* Bytes of fp32 workspace pa_paged_attention_decode needs for these sizes and `num_splits`
 * (0 = auto: the bound for any count the heuristic can pick). Host only. Layout inside:
 * partial accumulators [S, splits, Hq, D] then (m, l) pairs [S, splits, Hq, 2]. 0 when
 * one split suffices for every choice (then workspace may be NULL). */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int num_splits);

/* reshape_and_cache: for each token i with slot = slot_mapping[i] >= 0, copy key[i] to
 * k_cache[slot / block_size, slot % block_size] and value[i] likewise (bit-exact copy);
 * slot -1 writes nothing. Sources: "poot - Attention and KV Cache", KV cache (write map);
 * "32. Production attention kernels", Quantized KV caches (write_kv via slot_mapping).
 * key, value: [num_tokens, Hkv, D]; k_cache, v_cache: [num_blocks, block_size, Hkv, D];
 * slot_mapping: [num_tokens] int32. Two tokens naming one slot is the caller's error (the
 * result is one of them). A slot outside the pool is skipped and flagged. */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               void* k_cache, void* v_cache,
                               const int32_t* slot_mapping, int num_tokens,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               pa_dtype dtype, int32_t* error_word, void* stream);

/* reshape_and_cache with strided key/value rows: key row i starts key_row_stride elements after
 * row i - 1 (value likewise; 0 = dense, Hkv * D). Strides follow the pa_row_strides rules with
 * Hkv * D in place of Hq * D; everything else is pa_reshape_and_cache. */
pa_status pa_reshape_and_cache_strided(const void* key, const void* value, int64_t key_row_stride,
                                       int64_t value_row_stride, void* k_cache, void* v_cache,
                                       const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                                       int32_t* error_word, void* stream);

/* paged_attention_decode: one query per sequence, split-KV.
 * out[s, h] = softmax_p(scale * q[s,h] . K[s,p]) . V[s,p] over p in [0, context_lens[s]),
 * where K[s,p] = k_cache[block_tables[s, p / block_size], p % block_size, h / (Hq/Hkv)].
 * context_lens include the query's own (already cached) position; a zero length gives a
 * zero row. Sources: "paged-attn-xpu", Usage and Method; "TileInfer.jl - Attention
 * kernels", Decode: GQA packing and split-KV; "32. Production attention kernels", Long
 * contexts: split the keys.
 *   q [S, Hq, D], out [S, Hq, D] (dtype); block_tables [S, max_blocks_per_seq] int32;
 *   context_lens [S] int32; scale: 0 = 1/sqrt(D); num_splits: 0 = auto (heuristic above),
 *   else 1..32. workspace: device fp32 scratch of >= pa_decode_workspace_bytes(...) bytes
 *   (may be NULL when that is 0); it is fully overwritten, needs no initialisation, and must
 *   not be shared by calls that overlap on the GPU.
 * Supported: D in {64, 128, 256}; bf16 with Hq/Hkv <= 16 and block_size % 16 == 0;
 *   f32 with (Hq/Hkv) * D <= 2048 and any block_size >= 1. */
pa_status pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* context_lens,
                                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int num_blocks, int max_blocks_per_seq,
                                    float scale, pa_dtype dtype, int num_splits,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    int32_t* error_word, void* stream);

/* paged_attention_varlen: a flattened batch of R requests (prefill chunks, decodes and
 * verify blocks mixed). Request r owns query rows [query_start_loc[r], query_start_loc[r+1])
 * of q; its q_len queries are the newest q_len of its seq_lens[r] cached positions (query
 * t sits at position seq_lens[r] - q_len + t) and, when causal != 0, see keys at positions
 * <= their own; otherwise all seq_lens[r] keys. A query with no visible key gives zeros.
 * Sources: "32. Production attention kernels", One kernel for the whole batch;
 * "TileInfer.jl - Attention kernels", Prefill and Walking the block table.
 *   q, out [num_tokens, Hq, D]; query_start_loc [R+1] int32 (query_start_loc[R] must equal
 *   num_tokens); seq_lens [R] int32; block_tables [R, max_blocks_per_seq] int32;
 *   max_query_len: host upper bound on any q_len; it fixes the grid of the tensor-core path,
 *   whose rows past it are left unwritten and flagged (PA_ERRBIT_QUERY_LAYOUT).
 *   A request whose q_len exceeds its seq_len, or whose seq_len exceeds
 *   max_blocks_per_seq * block_size, gets zero rows and a flag.
 * Supported: D in {64, 128, 256}; bf16 with Hq/Hkv <= 16 and block_size % 16 == 0 (the
 *   tcgen05 tensor-core kernels serve every D with Hq/Hkv in {1,2,4,8,16} and block_size in
 *   {16,32,64,128}: at D 64 and 128 a CTA's two query tiles share each K/V tile, and a CTA
 *   whose second tile is empty (decodes, verify blocks) splits its key tiles between its two
 *   softmax groups; at D 256 it runs the two tiles one after the other; other bf16 shapes run
 *   every query token as a one-split decode); f32 with (Hq/Hkv) * D <= 2048 and any block_size. */
pa_status pa_paged_attention_varlen(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* query_start_loc, const int32_t* seq_lens,
                                    const int32_t* block_tables,
                                    int num_reqs, int num_tokens, int max_query_len,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int num_blocks, int max_blocks_per_seq,
                                    int causal, float scale, pa_dtype dtype,
                                    void* out, int32_t* error_word, void* stream);

/* pa_paged_attention_decode_static_scratch: the same decode, for callers that cannot allocate.
 * The pages describe no such variant; it exists for callers with no way to provide device
 * scratch: a plugin that its host framework gives only input and output pointers (no allocator,
 * no workspace hook), a runtime that has carved all device memory into its own pools and
 * forbids cudaMalloc after start-up, or a latency-bound loop that cannot pay cudaMalloc's
 * implicit device synchronisation.
 *   Arguments, layouts, results and supported shapes are those of pa_paged_attention_decode
 *   without `workspace` / `workspace_bytes`: the split partials go to a fixed 16 MiB
 *   (16,777,216-byte) array compiled into the library, which every GPU that loads the library
 *   holds until the process exits. The call allocates and frees nothing.
 *   - A batch whose partials need more than 16 MiB (units * splits * Hq * (D + 2) * 4 bytes,
 *     see pa_decode_workspace_bytes) is refused with PA_ERR_WORKSPACE_TOO_SMALL before
 *     anything is enqueued; pass a smaller num_splits (1 needs no scratch at all).
 *   - The first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 *     capture on that device. A failed lookup returns PA_ERR_CUDA. The address is kept for the
 *     life of the process and is not looked up again after a device reset (cudaDeviceReset or
 *     a re-created primary context): calling this entry point across a reset is unsupported.
 *   - Every call on a device shares the one array and it keeps the previous call's contents.
 *     Nothing in it needs to start at zero: each call writes every partial it later reads.
 *     Two calls that overlap on the GPU (e.g. on different streams) race on the array and give
 *     undefined results; serialise them. */
pa_status pa_paged_attention_decode_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                                   const int32_t* block_tables, const int32_t* context_lens,
                                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                                   int head_dim, int block_size, int num_blocks,
                                                   int max_blocks_per_seq, float scale, pa_dtype dtype,
                                                   int num_splits, void* out, int32_t* error_word,
                                                   void* stream);

/* pa_paged_attention_decode with score modifiers (see pa_attn_options; NULL = none). All other
 * arguments, layouts and rules are those of pa_paged_attention_decode. */
pa_status pa_paged_attention_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       float scale, pa_dtype dtype, int num_splits,
                                       void* out, void* workspace, size_t workspace_bytes,
                                       const pa_attn_options* options, int32_t* error_word, void* stream);

/* pa_paged_attention_decode_ex with strided q / out rows (see pa_row_strides; NULL = dense). */
pa_status pa_paged_attention_decode_strided(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables, const int32_t* context_lens,
                                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int num_blocks, int max_blocks_per_seq,
                                            float scale, pa_dtype dtype, int num_splits,
                                            void* out, void* workspace, size_t workspace_bytes,
                                            const pa_attn_options* options, const pa_row_strides* strides,
                                            int32_t* error_word, void* stream);

/* pa_paged_attention_varlen with score modifiers (see pa_attn_options; NULL = none). All other
 * arguments, layouts and rules are those of pa_paged_attention_varlen. */
pa_status pa_paged_attention_varlen_ex(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* query_start_loc, const int32_t* seq_lens,
                                       const int32_t* block_tables,
                                       int num_reqs, int num_tokens, int max_query_len,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       int causal, float scale, pa_dtype dtype,
                                       void* out, const pa_attn_options* options, int32_t* error_word,
                                       void* stream);

/* pa_paged_attention_varlen_ex with a workspace: pa_paged_attention_varlen_sched with
 * PA_SHORT_AUTO (NULL workspace: pa_paged_attention_varlen_ex). */
pa_status pa_paged_attention_varlen_ws(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* query_start_loc, const int32_t* seq_lens,
                                       const int32_t* block_tables,
                                       int num_reqs, int num_tokens, int max_query_len,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int max_blocks_per_seq,
                                       int causal, float scale, pa_dtype dtype,
                                       void* out, const pa_attn_options* options, void* workspace,
                                       size_t workspace_bytes, int32_t* error_word, void* stream);

/* pa_paged_attention_varlen_ws with strided q / out token rows (see pa_row_strides; NULL = dense).
 * The tensor-core path reads q through a tensor map whose token stride is strides->q. */
pa_status pa_paged_attention_varlen_strided(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* query_start_loc, const int32_t* seq_lens,
                                            const int32_t* block_tables,
                                            int num_reqs, int num_tokens, int max_query_len,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int num_blocks, int max_blocks_per_seq,
                                            int causal, float scale, pa_dtype dtype,
                                            void* out, const pa_attn_options* options,
                                            const pa_row_strides* strides, void* workspace,
                                            size_t workspace_bytes, int32_t* error_word, void* stream);

/* Where a varlen call with a workspace runs the batch's short requests (1 to 8 queries:
 * decodes and speculative verify blocks). */
typedef enum {
  PA_SHORT_AUTO = 0,   /* the split-KV decode for a batch of many short requests (num_reqs >= 80
                          and num_tokens <= 8 * num_reqs), else the tensor-core kernel (its decode
                          tiles then run beside the prefill tiles from the start; the split path's
                          extra launches only pay off over many short requests) */
  PA_SHORT_SPLIT = 1,  /* always the split-KV decode */
  PA_SHORT_TENSOR = 2  /* always the tensor-core kernel */
} pa_short_requests;

/* The varlen call on a grid planned on the device. The result is that of
 * pa_paged_attention_varlen (within the bf16 tolerance; bit for bit with PA_SHORT_TENSOR).
 * With a non-NULL workspace:
 *   - a one-CTA plan kernel reads query_start_loc and seq_lens on the device when the call runs
 *     and writes the batch's (tile pair, request) items, longest first by their key tiles, to the
 *     front of the workspace ("TileInfer.jl - Attention kernels", Open questions: heaviest causal
 *     blocks first); the tensor-core kernel, launched as its programmatic dependent, runs exactly
 *     those items on a grid of min(num_reqs * cdiv(max_query_len, 256 / G), num_tokens / (256 / G)
 *     + num_reqs) items x Hkv CTAs (the extra CTAs leave at once). Everything depends on host
 *     sizes and device buffers only, so a captured CUDA graph follows lengths and query layouts
 *     that change between replays;
 *   - short requests on the split-KV decode (per short_requests) are served by it, launched after
 *     the tensor-core grid as its programmatic dependent (its CTAs take the SMs that grid's tail
 *     frees), then its combine ("TileInfer.jl - Attention kernels", Decode: GQA packing and
 *     split-KV, the verify step; each query sees its own causal range).
 *   workspace: device memory of >= pa_varlen_workspace_bytes(...) bytes, 16-byte aligned, fully
 *   overwritten, not shared by calls that overlap on the GPU; PA_ERR_WORKSPACE_TOO_SMALL when
 *   shorter. NULL workspace: the default grid with every request on the tensor-core kernel
 *   (PA_SHORT_SPLIT then returns PA_ERR_WORKSPACE_TOO_SMALL). Up to four launches on `stream`.
 *   Other arguments, layouts and errors: pa_paged_attention_varlen_strided. bf16 shapes the
 *   tensor-core kernels serve; others run as pa_paged_attention_varlen (no workspace used). */
pa_status pa_paged_attention_varlen_sched(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* query_start_loc, const int32_t* seq_lens,
                                          const int32_t* block_tables,
                                          int num_reqs, int num_tokens, int max_query_len,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int max_blocks_per_seq,
                                          int causal, float scale, pa_dtype dtype,
                                          void* out, const pa_attn_options* options,
                                          const pa_row_strides* strides, pa_short_requests short_requests,
                                          void* workspace, size_t workspace_bytes, int32_t* error_word,
                                          void* stream);

/* ---------------------------------------------------------------------------------------
 * Planned varlen grid. The tensor-core kernel's default grid is every (query tile pair,
 * request, KV head) up to max_query_len, heaviest tile index first; CTAs of pairs a request does
 * not have exit at once but still take an SM slot (about 0.8 us each: 3,136 of the mixed
 * workload's 4,096 CTAs). A caller that knows its batch on the host (a serving engine builds
 * query_start_loc and seq_lens there) can plan instead: pa_varlen_plan lists only the pairs that
 * exist, longest first by their key tiles, and pa_paged_attention_varlen_planned runs exactly
 * those. ("TileInfer.jl - Attention kernels", Open questions: the heaviest causal blocks first.)
 * --------------------------------------------------------------------------------------- */

/* Upper bound on the items of a plan: cdiv(max_query_len, 2 * 128 / G) * num_reqs; -1 for bad
 * arguments (G = num_q_heads / num_kv_heads must be 1..16). Host only. */
int pa_varlen_plan_capacity(int num_reqs, int max_query_len, int num_q_heads, int num_kv_heads);

/* Host only: fill work_items (host memory, `capacity` entries) with the batch's (tile pair,
 * request) items, item = tile * num_reqs + request, ordered by descending key tiles of the
 * pair's longer tile. query_start_loc [num_reqs + 1] and seq_lens [num_reqs] are HOST copies of
 * what the call will read on the device; causal and sliding_window as in the call. Requests with
 * 1 <= q_len <= skip_upto are left out: pass 8 when the call gets a workspace (those requests then
 * go to the split-KV decode; see pa_paged_attention_varlen_ws), 0 otherwise. Returns the number of
 * items, or -1 for bad arguments or too small a capacity. The caller copies the items to the
 * device. */
int pa_varlen_plan(const int32_t* query_start_loc, const int32_t* seq_lens, int num_reqs, int max_query_len,
                   int num_q_heads, int num_kv_heads, int causal, int sliding_window, int skip_upto,
                   int32_t* work_items, int capacity);

/* pa_paged_attention_varlen_strided on a planned grid: work_items is a DEVICE copy of
 * pa_varlen_plan's output (num_items entries; NULL = pa_paged_attention_varlen_strided). With
 * work_items and a non-NULL workspace the short requests go to the split-KV decode (make the plan
 * with skip_upto 8), without a workspace to the tensor-core kernel. The plan must come from
 * the same batch: an item naming a tile past max_query_len is flagged (PA_ERRBIT_QUERY_LAYOUT)
 * and skipped, a request left out of the plan gets no rows. Same results as the default grid,
 * bit for bit (each pair's CTA computes the same thing, only the order changes). */
pa_status pa_paged_attention_varlen_planned(const void* q, const void* k_cache, const void* v_cache,
                                            const int32_t* query_start_loc, const int32_t* seq_lens,
                                            const int32_t* block_tables,
                                            int num_reqs, int num_tokens, int max_query_len,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, int num_blocks, int max_blocks_per_seq,
                                            int causal, float scale, pa_dtype dtype,
                                            void* out, const pa_attn_options* options,
                                            const pa_row_strides* strides, void* workspace,
                                            size_t workspace_bytes, const int32_t* work_items, int num_items,
                                            int32_t* error_word, void* stream);

/* Workspace bytes pa_paged_attention_varlen_ws / _sched need: the device-planned work list,
 * num_reqs * cdiv(max_blocks_per_seq * block_size, 16) int32 rounded up to 256 bytes, then the
 * split partials of num_reqs short requests (8 queries per request, at most 8 splits):
 * num_reqs * 8 * min(8, chunks) * Hq * (D + 2) * 4 with chunks = cdiv(max_blocks_per_seq *
 * block_size, 16), none when one split covers every context. 0 for num_reqs <= 0. Host only. */
size_t pa_varlen_workspace_bytes(int num_reqs, int num_q_heads, int head_dim, int max_blocks_per_seq,
                                 int block_size);

/* Self-test of the bounded waits inside the kernels (failure detection without a fault): a
 * one-thread kernel waits, with a limit of limit_us microseconds (1..1,000,000), on a barrier
 * that nothing ever completes, then ORs PA_ERRBIT_WAIT_TIMEOUT into *error_word (a device
 * int32) and returns, leaving the context usable. Every pipelined kernel waits through the
 * same helper with a 2-second limit. */
pa_status pa_selftest_wait_timeout(int limit_us, int32_t* error_word, void* stream);

/* ---------------------------------------------------------------------------------------
 * Cascade (shared-prefix) decode. "32. Production attention kernels", Long contexts: split the
 * keys (the same merge serves cascade attention: attend to a shared prefix once for many
 * requests, then merge with each request's own suffix) and Stretch exercises, item 2.
 * Sequence s's context is the prefix_len positions of the shared prefix (pages
 * prefix_table[0 .. cdiv(prefix_len, block_size))) followed by its own suffix_lens[s]
 * positions (pages suffix_tables[s, ...]); its one query is the last of them, so
 *   out[s, h] = softmax over prefix ++ suffix of (scale * q[s,h] . k) . v.
 * The prefix's K/V is read once for all sequences: a tensor-core pass puts all S * (Hq/Hkv)
 * query rows of a KV head against each key range of it (ranges sized to fill the SMs) and
 * writes their unnormalised partials; the suffixes run as the split-KV decode; the combine
 * merges all partials of a row by log-sum-exp. Three launches on `stream`; returns once they
 * are enqueued. Errors: as pa_paged_attention_decode (PA_ERR_WORKSPACE_TOO_SMALL for a short
 * workspace); a prefix_len outside [0, max_prefix_blocks * block_size] sets
 * PA_ERRBIT_LENGTH_OUT_OF_RANGE and is clamped.
 * --------------------------------------------------------------------------------------- */

/* Workspace bytes that suffice for pa_cascade_decode with these sizes and any split count. */
size_t pa_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int block_size,
                                  int max_prefix_blocks, int max_blocks_per_seq);

/*   q, out [S, Hq, D] bf16; k_cache, v_cache bf16 pools; prefix_table [max_prefix_blocks] int32;
 *   prefix_len: DEVICE int32 scalar (so a captured graph follows a growing prefix); suffix_tables
 *   [S, max_blocks_per_seq]; suffix_lens [S] (may be 0). num_splits: suffix splits (0 = auto, at most 31).
 *   workspace: >= pa_cascade_workspace_bytes, 16-byte aligned, device memory; the caller owns it.
 *   Supported: head_dim 64 or 128, Hq/Hkv in {1,2,4,8,16}, block_size in {16,32,64,128}. */
pa_status pa_cascade_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* prefix_table, const int32_t* prefix_len, int max_prefix_blocks,
                            const int32_t* suffix_tables, const int32_t* suffix_lens, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                            int max_blocks_per_seq, float scale, int num_splits, void* out, void* workspace,
                            size_t workspace_bytes, int32_t* error_word, void* stream);

/* ---------------------------------------------------------------------------------------
 * 8-bit KV cache. "32. Production attention kernels", Quantized KV caches; "TileInfer.jl -
 * Attention kernels", INT8 cache. The pools hold one code per element ([num_blocks,
 * block_size, Hkv, D], int8 or fp8 E4M3) and one float32 scale per (slot, KV head)
 * ([num_blocks, block_size, Hkv]); value = code * scale.
 * --------------------------------------------------------------------------------------- */

/* Quantise and write: for token i with slot = slot_mapping[i] >= 0 and each KV head, computed
 * in float32 exactly as the page does: amax = max(max_d |x|, 1e-8), scale = amax / q_max
 * (q_max 127 for PA_DTYPE_INT8, 448 for PA_DTYPE_FP8_E4M3), code = round-half-even(x / scale)
 * clamped to +-127 (int8) or x / scale rounded to nearest E4M3 (fp8); the codes go to
 * k_cache/v_cache[slot / block_size, slot % block_size] and the scale to k_scales/v_scales at
 * the same place. key, value: [num_tokens, Hkv, D] of src_dtype (bf16 or f32). Slot -1 writes
 * nothing; a slot outside the pool is skipped and flagged. head_dim must be a multiple of 32. */
pa_status pa_reshape_and_cache_quant(const void* key, const void* value, pa_dtype src_dtype,
                                     void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                     pa_dtype cache_dtype, const int32_t* slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                     int32_t* error_word, void* stream);

/* Decode over an 8-bit cache: as pa_paged_attention_decode_ex (q and out bf16), with keys and
 * values dequantised in registers: codes are converted exactly to fp16 (every int8 code and
 * every E4M3 value is an fp16 value) and the products run in fp16 with fp32 accumulation (q
 * converted to fp16, probabilities rounded to fp16); a key's scale multiplies its scores and a
 * value's scale its probabilities before P.V. int8 codes enter the products offset by 1152 (the
 * fp16 1152 + c, one byte permute per two codes) and the offsets are subtracted from the fp32
 * sums afterwards, which leaves those sums ~14 significant bits where fp32 has 24 (error of order
 * 1e-5 of the values' scale). Supported: D in {128, 256}, Hq/Hkv <= 16, block_size % 16 == 0. */
pa_status pa_paged_attention_decode_quant(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scales, const float* v_scales, pa_dtype cache_dtype,
                                          const int32_t* block_tables, const int32_t* context_lens,
                                          int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int max_blocks_per_seq,
                                          float scale, int num_splits, void* out, void* workspace,
                                          size_t workspace_bytes, const pa_attn_options* options,
                                          int32_t* error_word, void* stream);

/* Varlen over an 8-bit cache: as pa_paged_attention_varlen_ex (q and out bf16). At head_dim 128
 * with Hq/Hkv in {1,2,4,8,16} and block_size in {16,32,64,128} it runs on the tensor-core kernel:
 * each K / V tile's codes land in shared memory and are dequantised there to bf16 (code * scale,
 * rounded once to fp32 and then to bf16: "32. Production attention kernels", Quantized KV caches)
 * before the MMAs read them. Other shapes (head_dim 256) run every query token as a one-split
 * decode over the codes. Supported shapes as pa_paged_attention_decode_quant. */
pa_status pa_paged_attention_varlen_quant(const void* q, const void* k_cache, const void* v_cache,
                                          const float* k_scales, const float* v_scales, pa_dtype cache_dtype,
                                          const int32_t* query_start_loc, const int32_t* seq_lens,
                                          const int32_t* block_tables, int num_reqs, int num_tokens,
                                          int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, int max_blocks_per_seq, int causal,
                                          float scale, void* out, const pa_attn_options* options,
                                          int32_t* error_word, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* PAGED_ATTN_H_ */
