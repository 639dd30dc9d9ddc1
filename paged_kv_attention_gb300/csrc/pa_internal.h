// Internal host-side interface between the C-ABI entry points and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/paged_attn.h"

namespace pa {

constexpr int kMaxSplits = 32;
constexpr int kChunk = 16;  // tokens per decode pipeline stage

// Everything a decode-style kernel needs. A "unit" is one query row set that shares a
// context: a sequence (decode), a single query token of a varlen request (varlen generic
// path) or a group of consecutive queries of a short varlen request. Work is grid
// (unit * num_splits + split, kv head).
struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;     // decode: [units]
  const int32_t* query_start_loc;  // varlen: [num_reqs + 1]
  const int32_t* seq_lens;         // varlen: [num_reqs]
  void* out;
  float* ws_acc;  // [units, splits, Hq, D] when num_splits > 1
  float* ws_ml;   // [units, splits, Hq, 2]
  int32_t* err;
  // units: 0 = sequences (decode); 1 = the query tokens of varlen requests; 2 = groups of up to
  // unit_tokens consecutive queries of the varlen requests with 1 <= q_len <= small_max
  // (groups_per_req units per request; the other requests are skipped: nothing is written)
  int varlen;
  int unit_tokens;     // queries per unit (1 unless varlen == 2); rows = unit_tokens * group
  int groups_per_req;  // varlen == 2
  int small_max;       // varlen == 2
  int num_tokens;      // varlen == 2: rows of q / out (query blocks reaching past them are skipped)
  int causal;
  int num_reqs;
  int num_units;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int head_dim;
  int block_size;
  int num_blocks;
  int max_blocks;
  int num_splits;
  int chunks_per_split;
  float scale_log2;  // softmax scale * log2(e)
  // score modifiers (pa_attn_options)
  int window;            // > 0: a query at position t sees keys at positions > t - window
  float softcap_log2;    // > 0: score -> softcap * tanh(scale * s / softcap), in log2 units (* log2 e)
  float scale_over_cap;  // scale / softcap
  const float* sinks;    // nullable [Hq]: per-head sink logit (natural-log units)
  // 8-bit caches: 0 = bf16 values, 1 = int8 codes, 2 = fp8 E4M3 codes; scales [blocks, bs, Hkv]
  int quant;
  const float* k_scales;
  const float* v_scales;
  // partial-slot addressing: split `s` of unit `u` is slot u * slot_count + slot_offset + s;
  // force_partial writes partials even with one split (the cascade's suffix pass)
  int force_partial;
  int slot_offset;
  int slot_count;
  // elements from one query row (a sequence or token) of q / out to the next; 0 = dense (Hq * D)
  long long q_stride;
  long long out_stride;
  // 1: launched as a programmatic dependent of the previous kernel on the stream, which it does
  // not read from; its CTAs wait for that kernel's completion only before they exit, so that
  // this grid's completion implies the previous one's (the combine after it reads both)
  int overlap_previous;
  // balanced segments (8-bit caches, decode): CTAs per KV head, and the chunk offsets of the
  // sequences the decode grid leaves in the workspace for its combine
  int seg_ctas;
  int32_t* seg_off;
};

// key_stride / value_stride: bytes from one token's row to the next (multiples of 16)
cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int32_t* slot_mapping, int num_tokens, int row_bytes,
                                     long long key_stride, long long value_stride, long long num_slots,
                                     int32_t* err, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* err, cudaStream_t stream);

cudaError_t launch_reshape_and_cache_quant(const void* key, const void* value, bool src_bf16, void* k_cache,
                                           void* v_cache, float* k_scales, float* v_scales, bool fp8,
                                           const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                                           int head_dim, long long num_slots, int32_t* err, cudaStream_t stream);

// bf16 tensor-core decode (TMA page loads, mma.sync, 16-token chunks).
cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream);
int decode_bf16_ctas_per_sm(int head_dim, int group, int quant);

// fp32 CUDA-core decode.
cudaError_t launch_decode_f32(const DecodeParams& p, cudaStream_t stream);
int decode_f32_ctas_per_sm(int head_dim, int group);

// Balanced-segment decode over 8-bit caches (decode_seg.cu): every resident CTA of a KV head streams
// an equal share of the batch's chunks, followed by its combine. p.seg_ctas, ws_acc / ws_ml and
// seg_off must be set (see decode_seg_workspace_bytes).
bool decode_seg_supported(int head_dim, int group, int num_units, int quant);
int decode_seg_ctas_per_sm(int quant);
size_t decode_seg_workspace_bytes(int num_units, int num_q_heads, int ctas_per_head);
cudaError_t launch_decode_seg(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream);

// log-sum-exp merge of split partials into out.
cudaError_t launch_combine(const DecodeParams& p, pa_dtype dtype, cudaStream_t stream);

// tcgen05 varlen kernels (bf16; head_dim 64 and 128: two query tiles per CTA sharing every K/V
// tile; head_dim 256: the CTA's two query tiles one after the other).
struct VarlenParams {
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  void* out;
  int32_t* err;
  int num_reqs;
  int num_tokens;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int head_dim;
  int block_size;
  int num_blocks;
  int max_blocks;
  int max_query_len;
  int q_tiles;  // cdiv(max_query_len, tokens per CTA)
  int causal;
  float scale_log2;
  int window;
  float softcap_log2;
  float scale_over_cap;
  const float* sinks;
  // cascade prefix pass: all num_tokens query rows, non-causal over the prefix pages
  // (block_tables row 0) of length *prefix_len, cut into num_reqs key ranges of
  // prefix_tiles_per_split 128-key tiles; range r of row t writes its unnormalised partial to
  // slot t * slot_count + r of ws_acc / ws_ml instead of `out`
  int prefix_mode;
  const int32_t* prefix_len;
  // requests with 1 <= q_len <= skip_upto are left to the split-KV decode (launched beside this
  // kernel); 0 = none
  int skip_upto;
  int prefix_tiles_per_split;
  float* ws_acc;
  float* ws_ml;
  int slot_count;
  // elements from one token's output row to the next; 0 = dense (Hq * D). The query row stride
  // is carried by the query tensor map.
  long long out_stride;
  // planned grid: CTA i serves item work_items[i / num_kv_heads] = tile * num_reqs + request
  // (nullptr: every tile of every request, heaviest tile index first); a negative item is
  // padding and its CTAs leave at once
  const int32_t* work_items;
  int num_items;
  // 1: work_items is written by the plan kernel launched just before on the stream; this grid is
  // launched as its programmatic dependent and waits for it before reading the list
  int plan_on_device;
  // 8-bit caches (head_dim 128): 0 = bf16, 1 = int8 codes, 2 = fp8 E4M3 codes; one fp32 scale per
  // (slot, KV head) in k_scales / v_scales [blocks, bs, Hkv]
  int quant;
  const float* k_scales;
  const float* v_scales;
};
bool varlen_tc_supported(int head_dim, int group, int block_size);
// the cascade's prefix pass (two query tiles per CTA): head_dim 64 and 128
bool varlen_tc_prefix_supported(int head_dim, int group, int block_size);
// query tokens one CTA (work item) covers: two 128-row tiles of 128 / group tokens, any head_dim
int varlen_tc_tokens_per_cta(int group);
cudaError_t launch_varlen_tc(const VarlenParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream);
// Items the device-planned grid may hold for a batch of num_tokens queries in num_reqs requests
// (requests of at most skip_upto queries are left to the split-KV decode): the grid's size.
long long varlen_device_plan_capacity(int num_reqs, int num_tokens, int max_query_len, int group, int skip_upto);
// The device-side work list: `capacity` int32 entries of `items`, longest item first, -1 padded.
cudaError_t launch_varlen_device_plan(const int32_t* query_start_loc, const int32_t* seq_lens, int num_reqs,
                                      int num_tokens, int group, int q_tiles, int causal, int window, int skip_upto,
                                      int32_t* items, int capacity, int32_t* err, cudaStream_t stream);
// head_dim 256 (in varlen_tc256.cu); `ctas` already checked against the grid limit
cudaError_t launch_varlen_tc256(const VarlenParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, long long ctas, cudaStream_t stream);

}  // namespace pa
