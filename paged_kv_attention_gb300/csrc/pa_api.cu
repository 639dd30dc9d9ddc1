// C-ABI entry points: argument validation, split planning, TMA descriptor encoding and
// launches on the caller's stream. Nothing here allocates device memory or synchronises.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_head_dim(int d) { return d == 64 || d == 128 || d == 256; }
long long cdivll(long long a, long long b) { return (a + b - 1) / b; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// [num_blocks, block_size, Hkv, D] pool (bf16, or 8-bit codes when elt == 1) viewed as a 4-D
// tensor (D, Hkv, bs, blocks); one box is `box_tokens` rows of one KV head, 128 bytes wide
// (64 bf16 or 128 codes), 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int D, int Hkv, int bs, int num_blocks, int box_tokens,
                      int elt = 2) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)bs, (cuuint64_t)num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)D * elt, (cuuint64_t)Hkv * D * elt, (cuuint64_t)bs * Hkv * D * elt};
  cuuint32_t box[4] = {(cuuint32_t)(128 / elt), 1, (cuuint32_t)box_tokens, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same bf16 pool viewed as a 5-D tensor (64 columns, 8 rows, D / 64 column blocks, row
// groups of 8 across the pool, Hkv) so that one box is a whole page of one KV head (bs <= 128
// rows, every column block) landing as [row group][column block][8 rows x 128 bytes]: one copy
// per page instead of one per 64-column block. Each 8-row x 128-byte block is a 128-byte-swizzle
// atom; row groups sit 256 * D / 64 bytes apart, column blocks 1,024 bytes apart.
bool encode_cache_map_pages(CUtensorMap* map, const void* base, int D, int Hkv, int bs, int num_blocks) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || bs % 8 != 0 || bs > 128 || D % 64 != 0) return false;
  const cuuint64_t row = (cuuint64_t)Hkv * D * 2;
  cuuint64_t dims[5] = {64, 8, (cuuint64_t)D / 64, (cuuint64_t)num_blocks * bs / 8, (cuuint64_t)Hkv};
  cuuint64_t strides[4] = {row, 128, 8 * row, (cuuint64_t)D * 2};
  cuuint32_t box[5] = {64, 8, (cuuint32_t)D / 64, (cuuint32_t)bs / 8, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The split-KV decode's K / V maps: one box is `box_tokens` rows of one KV head over every
// 128-byte column of the row, landing as [column][row][128 bytes] (the 4-D map's boxes, one copy
// instead of one per column). The pool viewed as (128-byte columns' elements, bs, columns, Hkv,
// blocks).
bool encode_decode_cache_map(CUtensorMap* map, const void* base, int D, int Hkv, int bs, int num_blocks,
                             int box_tokens, int elt = 2) {
  const int cols = D * elt / 128;
  if (cols <= 1) return encode_cache_map(map, base, D, Hkv, bs, num_blocks, box_tokens, elt);
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[5] = {(cuuint64_t)(128 / elt), (cuuint64_t)bs, (cuuint64_t)cols, (cuuint64_t)Hkv,
                        (cuuint64_t)num_blocks};
  cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * elt, 128, (cuuint64_t)D * elt, (cuuint64_t)bs * Hkv * D * elt};
  cuuint32_t box[5] = {(cuuint32_t)(128 / elt), (cuuint32_t)box_tokens, (cuuint32_t)cols, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The bf16 K / V maps of the tensor-core varlen kernels: whole-page boxes at head_dim 128, one
// box per page and 64-column block otherwise (head_dim 64 has one block; the head_dim-256 kernel
// keeps its own layout).
bool encode_varlen_cache_map(CUtensorMap* map, const void* base, int D, int Hkv, int bs, int num_blocks) {
  if (D == 128) return encode_cache_map_pages(map, base, D, Hkv, bs < 128 ? bs : 128, num_blocks);
  return encode_cache_map(map, base, D, Hkv, bs, num_blocks, bs < 128 ? bs : 128);
}

// q [N, Hq, D] bf16 (rows row_stride elements apart) viewed as (D, Hq, N); one box = `tokens`
// tokens x `group` heads x 64 cols.
bool encode_query_map(CUtensorMap* map, const void* base, int D, int Hq, int N, int group, int tokens,
                      long long row_stride) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)row_stride * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Per-device facts, filled lazily. The occupancy slots are written by whichever host thread
// first needs them (every writer stores the same value), so they are atomics.
struct DeviceInfo {
  int sms = 0;
  std::atomic<int> occ_bf16[3][3][2] = {};  // [bf16 | int8 | fp8][D 64/128/256][group <= 8 | > 8]
  std::atomic<int> occ_f32[3][5] = {};      // [D][padded group 1..16]
};

bool device_info(DeviceInfo** out) {
  static DeviceInfo infos[64];
  static bool ready[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    if (cudaDeviceGetAttribute(&infos[dev].sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    ready[dev] = true;
  }
  *out = &infos[dev];
  return true;
}

int dim_index(int d) { return d == 64 ? 0 : (d == 128 ? 1 : 2); }
int log2i(int g) {
  int l = 0;
  while ((1 << l) < g) ++l;
  return l;
}

bool group_ok_bf16(int G) { return G >= 1 && G <= 16; }
bool group_ok_f32(int G, int D) { return G >= 1 && G <= 16 && G * D <= 2048; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// A caller's row stride in elements: 0 = dense rows; otherwise at least a dense row (rows never
// overlap) and a whole number of 16-byte units, so every row stays 16-byte aligned.
bool resolve_row_stride(long long given, long long dense, int elt, long long* out) {
  if (given == 0) {
    *out = dense;
    return true;
  }
  if (given < dense || (given * elt) % 16 != 0 || given > (1ll << 36)) return false;
  *out = given;
  return true;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARGUMENT: return "PA_ERR_INVALID_ARGUMENT";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "PA_ERR_WORKSPACE_TOO_SMALL";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    default: return "PA_ERR_UNKNOWN";
  }
}

extern "C" int pa_version(void) { return kVersion; }

extern "C" int pa_supports(int is_varlen, int head_dim, int num_q_heads, int num_kv_heads, int block_size,
                           pa_dtype dtype) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0) return 0;
  if (!valid_head_dim(head_dim)) return 0;
  const int G = num_q_heads / num_kv_heads;
  if (dtype == PA_DTYPE_BF16) return group_ok_bf16(G) && block_size % kChunk == 0 ? 1 : 0;
  if (dtype == PA_DTYPE_F32) return group_ok_f32(G, head_dim) ? 1 : 0;
  (void)is_varlen;
  return 0;
}

extern "C" int pa_plan_decode_splits(int num_units, int max_chunks, int num_sms, int ctas_per_sm,
                                     int min_chunks_per_split) {
  if (num_units <= 0 || max_chunks <= 0 || num_sms <= 0 || ctas_per_sm <= 0) return 1;
  // Never a split under 4 chunks (64 tokens), none at all past 32, never more splits than
  // chunks. Each CTA pays a fixed start-up and merge cost, so splits should be long: prefer
  // splits of at least `min_chunks_per_split` chunks, unless that leaves less than one wave of
  // resident CTAs, in which case split (down to 4 chunks) until one wave is filled.
  constexpr int kMinChunksPerSplit = 4;
  const long long slots = (long long)num_sms * ctas_per_sm;
  const long long cap = std::max<long long>(1, std::min<long long>(kMaxSplits, max_chunks / kMinChunksPerSplit));
  const long long cap_long = std::max<long long>(1, std::min<long long>(cap, max_chunks / std::max(1, min_chunks_per_split)));
  const long long fill = cdivll(slots, num_units);  // splits for one full wave
  if (fill > cap_long) return (int)std::min<long long>(fill, cap);
  // among the long enough counts, the one whose CTA count best fills whole waves; a larger
  // count must fill them clearly better to win
  int best = 1;
  double best_eff = -1.0;
  for (int sp = 1; sp <= cap_long; ++sp) {
    // splits whose boundaries fall on the same chunks are one choice: keep the smallest
    const long long per = cdivll(max_chunks, sp);
    if (cdivll(max_chunks, per) != sp) continue;
    const long long ctas = (long long)num_units * sp;
    const long long waves = cdivll(ctas, slots);
    const double eff = (double)ctas / (double)(waves * slots);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = sp;
    }
  }
  return best;
}

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_blocks_per_seq,
                                            int block_size, int num_splits) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0) return 0;
  const long long max_chunks = cdivll((long long)max_blocks_per_seq * block_size, kChunk);
  long long splits;
  if (num_splits <= 0) {
    splits = std::min<long long>(kMaxSplits, std::max<long long>(1, max_chunks / 4));
  } else {
    splits = std::min<long long>(num_splits, max_chunks);
  }
  if (splits <= 1) return 0;
  const long long per_slot = (long long)head_dim + 2;
  return (size_t)((long long)num_seqs * splits * num_q_heads * per_slot * 4);
}

extern "C" pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                          const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                                          int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                                          int32_t* error_word, void* stream) {
  return pa_reshape_and_cache_strided(key, value, 0, 0, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads,
                                      head_dim, block_size, num_blocks, dtype, error_word, stream);
}

extern "C" pa_status pa_reshape_and_cache_strided(const void* key, const void* value, int64_t key_row_stride,
                                                  int64_t value_row_stride, void* k_cache, void* v_cache,
                                                  const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                                                  int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                                                  int32_t* error_word, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARGUMENT;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARGUMENT;
  const int elem = dtype == PA_DTYPE_BF16 ? 2 : 4;
  const long long row_bytes = (long long)num_kv_heads * head_dim * elem;
  if (row_bytes % 16 != 0 || row_bytes > (1ll << 30)) return PA_ERR_UNSUPPORTED;
  const long long row_elems = (long long)num_kv_heads * head_dim;
  long long key_stride = 0, value_stride = 0;
  if (!resolve_row_stride(key_row_stride, row_elems, elem, &key_stride) ||
      !resolve_row_stride(value_row_stride, row_elems, elem, &value_stride))
    return PA_ERR_INVALID_ARGUMENT;
  const long long num_slots = (long long)num_blocks * block_size;
  cudaError_t e = launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens, (int)row_bytes,
                                           key_stride * elem, value_stride * elem, num_slots, error_word,
                                           as_stream(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace {

pa_status validate_common(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          const void* out, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, int max_blocks_per_seq, float scale, pa_dtype dtype) {
  if (!q || !k_cache || !v_cache || !block_tables || !out) return PA_ERR_INVALID_ARGUMENT;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARGUMENT;
  if (head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (!(scale >= 0.f) || isinf(scale)) return PA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID_ARGUMENT;
  if ((long long)max_blocks_per_seq * block_size > (1ll << 30)) return PA_ERR_UNSUPPORTED;
  if (dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
  if (!valid_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (dtype == PA_DTYPE_BF16 && (!group_ok_bf16(G) || block_size % kChunk != 0)) return PA_ERR_UNSUPPORTED;
  if (dtype == PA_DTYPE_F32 && !group_ok_f32(G, head_dim)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Preferred shortest split, in 16-token chunks (measured on GB300 at 64 x 4096: bf16 calls ran
// 171 us at the wave-filling 7 splits and 167 us at 3-4; 8-bit-code calls, limited by their
// consumers rather than HBM, 160 us at 7 splits and 112-113 us at 1).
constexpr int kMinChunksPerSplitBf16 = 64;
constexpr int kMinChunksPerSplitCodes = 256;

// Varlen requests of at most this many queries (decodes, speculative verify blocks) go to the
// split-KV decode when the caller gives pa_paged_attention_varlen_ws a workspace; they run as
// units of up to 8 query rows (unit_tokens queries x group: one MMA n-tile) with at most 8
// splits. (Units of 16 rows, two n-tiles, read a verify block's keys fewer times but measured
// slower: 48 vs 46 us for 8 verify blocks of 5 queries, 103 vs 87 us for 48 decodes.)
constexpr int kShortRequestQueries = 8;
constexpr int kShortRequestMaxSplits = 8;
int short_unit_tokens(int G) { return std::min(kShortRequestQueries, std::max(1, 8 / G)); }

int auto_splits(DeviceInfo* info, int units, int Hkv, int D, int G, long long max_chunks, pa_dtype dtype,
                int quant = 0) {
  int occ;
  if (dtype == PA_DTYPE_BF16 || quant != 0) {
    std::atomic<int>& slot = info->occ_bf16[quant][dim_index(D)][G > 8 ? 1 : 0];
    occ = slot.load(std::memory_order_relaxed);
    if (occ == 0) {
      occ = decode_bf16_ctas_per_sm(D, G, quant);
      slot.store(occ, std::memory_order_relaxed);
    }
  } else {
    std::atomic<int>& slot = info->occ_f32[dim_index(D)][log2i(G)];
    occ = slot.load(std::memory_order_relaxed);
    if (occ == 0) {
      occ = decode_f32_ctas_per_sm(D, G);
      slot.store(occ, std::memory_order_relaxed);
    }
  }
  int s = pa_plan_decode_splits(units * Hkv, (int)std::min<long long>(max_chunks, 1 << 30), info->sms, occ,
                                quant != 0 ? kMinChunksPerSplitCodes : kMinChunksPerSplitBf16);
  s = (int)std::min<long long>(s, max_chunks);
  const long long per = cdivll(max_chunks, s);
  return (int)cdivll(max_chunks, per);
}

// Bytes at the front of a varlen workspace that hold the device-planned work list: room for
// every tile pair the grid could index, num_reqs * cdiv(max_query_len, 16) (a CTA covers at least
// 16 queries), rounded up to 256 bytes.
size_t varlen_plan_bytes(int num_reqs, int max_query_len) {
  const long long items = (long long)num_reqs * cdivll(std::max(max_query_len, 1), 16);
  return (size_t)cdivll(items * 4, 256) * 256;
}

// Split count and partial layout of run_decode_units (without launching): the plan it will make.
int decode_units_splits(const DecodeParams& p, pa_dtype dtype, int requested_splits, DeviceInfo* info);

// Launch the decode-style kernels over `p.num_units` units (already filled in except the
// split fields), then the combine when splitting.
int decode_units_splits(const DecodeParams& p, pa_dtype dtype, int requested_splits, DeviceInfo* info) {
  const long long max_chunks = cdivll((long long)p.max_blocks * p.block_size, kChunk);
  const int T = std::max(1, p.unit_tokens);  // queries per unit; the kernel's rows are T * group
  int splits = requested_splits;
  if (splits <= 0)
    splits = auto_splits(info, p.num_units, p.num_kv_heads, p.head_dim, p.group * T, max_chunks, dtype, p.quant);
  if (p.varlen == 2) splits = std::min(splits, kShortRequestMaxSplits);
  splits = (int)std::min<long long>(splits, max_chunks);
  const int per = (int)cdivll(max_chunks, splits);
  return (int)cdivll(max_chunks, per);
}

// The workspace check of run_decode_units (auto splits), done before the varlen call launches
// anything: a refused call must enqueue nothing.
pa_status check_decode_units_workspace(const DecodeParams& p, const void* workspace, size_t workspace_bytes) {
  DeviceInfo* info = nullptr;
  if (!device_info(&info)) return PA_ERR_CUDA;
  const int splits = decode_units_splits(p, PA_DTYPE_BF16, 0, info);
  if (splits <= 1) return PA_OK;
  const size_t need = (size_t)p.num_units * splits * std::max(1, p.unit_tokens) * p.num_q_heads *
                      ((size_t)p.head_dim + 2) * 4;
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return PA_ERR_INVALID_ARGUMENT;
  return PA_OK;
}

pa_status run_decode_units(DecodeParams& p, pa_dtype dtype, const void* k_cache, const void* v_cache,
                           int requested_splits, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  DeviceInfo* info = nullptr;
  if (!device_info(&info)) return PA_ERR_CUDA;
  const int D = p.head_dim;
  const long long max_chunks = cdivll((long long)p.max_blocks * p.block_size, kChunk);
  const int T = std::max(1, p.unit_tokens);  // queries per unit; the kernel's rows are T * group
  const int splits = decode_units_splits(p, dtype, requested_splits, info);
  const int per = (int)cdivll(max_chunks, splits);
  p.num_splits = splits;
  p.chunks_per_split = per;
  p.slot_count = splits;
  p.slot_offset = 0;
  p.force_partial = 0;
  if (splits > 1) {
    const size_t slots = (size_t)p.num_units * splits * T * p.num_q_heads;
    const size_t need = slots * ((size_t)D + 2) * 4;
    if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return PA_ERR_INVALID_ARGUMENT;
    p.ws_acc = static_cast<float*>(workspace);
    p.ws_ml = p.ws_acc + slots * D;
  }
  cudaError_t e;
  if (dtype == PA_DTYPE_BF16 || p.quant != 0) {
    const int elt = p.quant != 0 ? 1 : 2;
    CUtensorMap kmap, vmap;
    if (!encode_decode_cache_map(&kmap, k_cache, D, p.num_kv_heads, p.block_size, p.num_blocks, kChunk, elt) ||
        !encode_decode_cache_map(&vmap, v_cache, D, p.num_kv_heads, p.block_size, p.num_blocks, kChunk, elt))
      return PA_ERR_CUDA;
    e = launch_decode_bf16(p, kmap, vmap, stream);
  } else {
    e = launch_decode_f32(p, stream);
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (splits > 1) {
    e = launch_combine(p, p.quant != 0 ? PA_DTYPE_BF16 : dtype, stream);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_auto_splits(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                     int max_blocks_per_seq, pa_dtype dtype) {
  if (num_seqs <= 0) return 0;
  static const int dummy[4] __attribute__((aligned(16))) = {};
  if (validate_common(dummy, dummy, dummy, dummy, dummy, num_q_heads, num_kv_heads, head_dim, block_size, 1,
                      max_blocks_per_seq, 0.f, dtype) != PA_OK)
    return 0;
  DeviceInfo* info = nullptr;
  if (!device_info(&info)) return 0;
  const long long max_chunks = cdivll((long long)max_blocks_per_seq * block_size, kChunk);
  return auto_splits(info, num_seqs, num_kv_heads, head_dim, num_q_heads / num_kv_heads, max_chunks, dtype);
}

namespace {

// Checks and applies pa_attn_options (NULL = none) to the score-modifier fields of p.
template <typename Params>
pa_status apply_options(const pa_attn_options* o, float scale, Params& p) {
  p.window = 0;
  p.softcap_log2 = 0.f;
  p.scale_over_cap = 0.f;
  p.sinks = nullptr;
  if (o == nullptr) return PA_OK;
  if (o->sliding_window < 0) return PA_ERR_INVALID_ARGUMENT;
  if (!(o->logit_softcap >= 0.f) || isinf(o->logit_softcap)) return PA_ERR_INVALID_ARGUMENT;
  if (o->sinks != nullptr && (reinterpret_cast<uintptr_t>(o->sinks) & 3u) != 0) return PA_ERR_INVALID_ARGUMENT;
  p.window = o->sliding_window;
  if (o->logit_softcap > 0.f) {
    p.softcap_log2 = o->logit_softcap * kLog2e;
    p.scale_over_cap = scale / o->logit_softcap;
  }
  p.sinks = o->sinks;
  return PA_OK;
}

// The q / out row strides of a pa_row_strides (NULL = dense rows), checked.
bool resolve_strides(const pa_row_strides* st, int num_q_heads, int head_dim, pa_dtype dtype, long long* q_stride,
                     long long* out_stride) {
  const long long dense = (long long)num_q_heads * head_dim;
  const int elt = dtype == PA_DTYPE_F32 ? 4 : 2;
  return resolve_row_stride(st ? st->q : 0, dense, elt, q_stride) &&
         resolve_row_stride(st ? st->out : 0, dense, elt, out_stride);
}

}  // namespace

extern "C" pa_status pa_paged_attention_decode(const void* q, const void* k_cache, const void* v_cache,
                                               const int32_t* block_tables, const int32_t* context_lens,
                                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                               int block_size, int num_blocks, int max_blocks_per_seq, float scale,
                                               pa_dtype dtype, int num_splits, void* out, void* workspace,
                                               size_t workspace_bytes, int32_t* error_word, void* stream) {
  return pa_paged_attention_decode_ex(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                      num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale,
                                      dtype, num_splits, out, workspace, workspace_bytes, nullptr, error_word,
                                      stream);
}

extern "C" pa_status pa_paged_attention_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                                  float scale, pa_dtype dtype, int num_splits, void* out,
                                                  void* workspace, size_t workspace_bytes,
                                                  const pa_attn_options* options, int32_t* error_word,
                                                  void* stream) {
  return pa_paged_attention_decode_strided(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                           num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale,
                                           dtype, num_splits, out, workspace, workspace_bytes, options, nullptr,
                                           error_word, stream);
}

extern "C" pa_status pa_paged_attention_decode_strided(const void* q, const void* k_cache, const void* v_cache,
                                                       const int32_t* block_tables, const int32_t* context_lens,
                                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                                       int head_dim, int block_size, int num_blocks,
                                                       int max_blocks_per_seq, float scale, pa_dtype dtype,
                                                       int num_splits, void* out, void* workspace,
                                                       size_t workspace_bytes, const pa_attn_options* options,
                                                       const pa_row_strides* strides, int32_t* error_word,
                                                       void* stream) {
  if (num_seqs < 0 || num_splits < 0 || num_splits > kMaxSplits) return PA_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PA_OK;
  if (!context_lens) return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_common(q, k_cache, v_cache, block_tables, out, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, scale, dtype);
  if (st != PA_OK) return st;
  long long q_stride = 0, out_stride = 0;
  if (!resolve_strides(strides, num_q_heads, head_dim, dtype, &q_stride, &out_stride)) return PA_ERR_INVALID_ARGUMENT;
  if ((long long)num_seqs * num_kv_heads * kMaxSplits > (1ll << 31) - 1) return PA_ERR_UNSUPPORTED;
  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = error_word;
  p.varlen = 0;
  p.causal = 0;
  p.num_units = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.q_stride = q_stride;
  p.out_stride = out_stride;
  const float sc = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;
  p.scale_log2 = sc * kLog2e;
  st = apply_options(options, sc, p);
  if (st != PA_OK) return st;
  return run_decode_units(p, dtype, k_cache, v_cache, num_splits, workspace, workspace_bytes, as_stream(stream));
}

extern "C" pa_status pa_paged_attention_varlen(const void* q, const void* k_cache, const void* v_cache,
                                               const int32_t* query_start_loc, const int32_t* seq_lens,
                                               const int32_t* block_tables, int num_reqs, int num_tokens,
                                               int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                                               int block_size, int num_blocks, int max_blocks_per_seq, int causal,
                                               float scale, pa_dtype dtype, void* out, int32_t* error_word,
                                               void* stream) {
  return pa_paged_attention_varlen_ex(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs,
                                      num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, max_blocks_per_seq, causal, scale, dtype, out, nullptr,
                                      error_word, stream);
}

extern "C" size_t pa_varlen_workspace_bytes(int num_reqs, int num_q_heads, int head_dim, int max_blocks_per_seq,
                                            int block_size) {
  // units x queries per unit = num_reqs x kShortRequestQueries for every group size (the unit
  // sizes divide it), at most kShortRequestMaxSplits splits
  if (num_reqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0) return 0;
  const long long max_chunks = cdivll((long long)max_blocks_per_seq * block_size, kChunk);
  const long long splits = std::min<long long>(kShortRequestMaxSplits, max_chunks);
  // the device-planned work list first (a query length never exceeds the table's capacity)
  const long long max_q = std::min<long long>((long long)max_blocks_per_seq * block_size, 1ll << 30);
  const size_t plan = varlen_plan_bytes(num_reqs, (int)max_q);
  if (splits <= 1) return plan;
  return plan +
         (size_t)((long long)num_reqs * kShortRequestQueries * splits * num_q_heads * ((long long)head_dim + 2) * 4);
}

extern "C" pa_status pa_paged_attention_varlen_ex(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* query_start_loc, const int32_t* seq_lens,
                                                  const int32_t* block_tables, int num_reqs, int num_tokens,
                                                  int max_query_len, int num_q_heads, int num_kv_heads,
                                                  int head_dim, int block_size, int num_blocks,
                                                  int max_blocks_per_seq, int causal, float scale, pa_dtype dtype,
                                                  void* out, const pa_attn_options* options, int32_t* error_word,
                                                  void* stream) {
  return pa_paged_attention_varlen_ws(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs,
                                      num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, max_blocks_per_seq, causal, scale, dtype, out, options, nullptr, 0,
                                      error_word, stream);
}

extern "C" pa_status pa_paged_attention_varlen_ws(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* query_start_loc, const int32_t* seq_lens,
                                                  const int32_t* block_tables, int num_reqs, int num_tokens,
                                                  int max_query_len, int num_q_heads, int num_kv_heads,
                                                  int head_dim, int block_size, int num_blocks,
                                                  int max_blocks_per_seq, int causal, float scale, pa_dtype dtype,
                                                  void* out, const pa_attn_options* options, void* workspace,
                                                  size_t workspace_bytes, int32_t* error_word, void* stream) {
  return pa_paged_attention_varlen_strided(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs,
                                           num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim,
                                           block_size, num_blocks, max_blocks_per_seq, causal, scale, dtype, out,
                                           options, nullptr, workspace, workspace_bytes, error_word, stream);
}

extern "C" pa_status pa_paged_attention_varlen_strided(const void* q, const void* k_cache, const void* v_cache,
                                                       const int32_t* query_start_loc, const int32_t* seq_lens,
                                                       const int32_t* block_tables, int num_reqs, int num_tokens,
                                                       int max_query_len, int num_q_heads, int num_kv_heads,
                                                       int head_dim, int block_size, int num_blocks,
                                                       int max_blocks_per_seq, int causal, float scale,
                                                       pa_dtype dtype, void* out, const pa_attn_options* options,
                                                       const pa_row_strides* strides, void* workspace,
                                                       size_t workspace_bytes, int32_t* error_word, void* stream) {
  return pa_paged_attention_varlen_planned(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs,
                                           num_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim,
                                           block_size, num_blocks, max_blocks_per_seq, causal, scale, dtype, out,
                                           options, strides, workspace, workspace_bytes, nullptr, -1, error_word,
                                           stream);
}

extern "C" int pa_varlen_plan_capacity(int num_reqs, int max_query_len, int num_q_heads, int num_kv_heads) {
  if (num_reqs < 0 || max_query_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return -1;
  const int G = num_q_heads / num_kv_heads;
  if (G > 16) return -1;
  const long long n = cdivll(max_query_len, varlen_tc_tokens_per_cta(G)) * (long long)num_reqs;
  return n > (1ll << 31) - 1 ? -1 : (int)n;
}

extern "C" int pa_varlen_plan(const int32_t* query_start_loc, const int32_t* seq_lens, int num_reqs,
                              int max_query_len, int num_q_heads, int num_kv_heads, int causal, int sliding_window,
                              int skip_upto, int32_t* work_items, int capacity) {
  const int cap_needed = pa_varlen_plan_capacity(num_reqs, max_query_len, num_q_heads, num_kv_heads);
  if (cap_needed < 0 || sliding_window < 0 || skip_upto < 0 || capacity < 0) return -1;
  if (num_reqs == 0) return 0;
  if (!query_start_loc || !seq_lens || !work_items) return -1;
  const int G = num_q_heads / num_kv_heads;
  const int TOK = 128 / G;                       // tokens of one 128-row query tile
  const int per_cta = varlen_tc_tokens_per_cta(G);  // a CTA's two tiles
  const int q_tiles = (int)cdivll(max_query_len, per_cta);
  // key tiles (128 keys) the query tile [tok0, tok0 + n) of a request walks
  auto key_tiles = [&](int q_len, int seq, int tok0) {
    const int n = std::max(0, std::min(TOK, q_len - tok0));
    if (n == 0) return 0;
    const int first = seq - q_len + tok0;
    const int key_end = causal ? std::min(seq, first + n) : seq;
    const int j0 = sliding_window > 0 ? std::max(0, first - sliding_window + 1) / 128 : 0;
    return std::max(0, (int)cdivll(std::max(0, key_end), 128) - j0);
  };
  struct Item {
    int work;
    int32_t id;
  };
  std::vector<Item> items;
  for (int r = 0; r < num_reqs; ++r) {
    const int q_len = query_start_loc[r + 1] - query_start_loc[r];
    if (q_len <= 0 || q_len <= skip_upto) continue;  // nothing here, or served by the split-KV decode
    const int seq = seq_lens[r];
    const int tiles = std::min((int)cdivll(q_len, per_cta), q_tiles);
    for (int t = 0; t < tiles; ++t) {
      const int tok0 = t * per_cta;
      const int work = std::max(key_tiles(q_len, seq, tok0), key_tiles(q_len, seq, tok0 + TOK));
      items.push_back({work, (int32_t)(t * num_reqs + r)});
    }
  }
  if ((long long)items.size() > capacity) return -1;
  // longest first (a CTA's time is about proportional to its key tiles), ties in request order
  std::stable_sort(items.begin(), items.end(), [](const Item& a, const Item& b) { return a.work > b.work; });
  for (size_t i = 0; i < items.size(); ++i) work_items[i] = items[i].id;
  return (int)items.size();
}

namespace pa {
namespace {
// PA_SHORT_AUTO sends the short requests to the split-KV decode when the batch has at least
// kAutoSplitMinReqs requests averaging at most kAutoSplitMaxAvgQueries queries. The split path adds
// a launch chain (plan, tensor-core grid, decode, combine: ~10 us) that only many short requests
// repay, while on the tensor-core grid decode tiles run beside the prefill tiles from the start.
// Measured on GB300 (us, device-planned tensor-core grid vs split, L2 cold; contexts up to 4,096,
// chunks of 512, verify blocks of 5): 8 chunks + 48 decodes + 8 verify blocks 182 vs 203; 48
// decodes + 8 verify 103 vs 113; 2 chunks + 48 decodes + 8 verify 132 vs 142; 1 chunk + 64
// decodes 115 vs 117; 4 chunks + 128 decodes 250 vs 252; 48 decodes 91 vs 95; 64 decodes 108 vs
// 110; 96 decodes 149 vs 145; 128 decodes 203 vs 189; 120 decodes + 8 verify 205 vs 194; 1 chunk +
// 256 decodes 396 vs 373; 256 decodes 404 vs 353; 512 decodes 744 vs 630.
constexpr int kAutoSplitMinReqs = 80;
constexpr int kAutoSplitMaxAvgQueries = 8;

pa_status varlen_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* query_start_loc,
                      const int32_t* seq_lens, const int32_t* block_tables, int num_reqs, int num_tokens,
                      int max_query_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, int max_blocks_per_seq, int causal, float scale, pa_dtype dtype, void* out,
                      const pa_attn_options* options, const pa_row_strides* strides, int short_requests,
                      void* workspace, size_t workspace_bytes, const int32_t* work_items, int num_items,
                      int32_t* error_word, void* stream) {
  if (short_requests < PA_SHORT_AUTO || short_requests > PA_SHORT_TENSOR) return PA_ERR_INVALID_ARGUMENT;
  if (num_reqs < 0 || num_tokens < 0 || max_query_len < 0) return PA_ERR_INVALID_ARGUMENT;
  if (work_items != nullptr && num_items < 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_reqs == 0 || num_tokens == 0) return PA_OK;
  if (!query_start_loc || !seq_lens) return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_common(q, k_cache, v_cache, block_tables, out, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, scale, dtype);
  if (st != PA_OK) return st;
  long long q_stride = 0, out_stride = 0;
  if (!resolve_strides(strides, num_q_heads, head_dim, dtype, &q_stride, &out_stride)) return PA_ERR_INVALID_ARGUMENT;
  if ((long long)num_tokens * num_kv_heads > (1ll << 31) - 1) return PA_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  const float sc = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;
  cudaStream_t s = as_stream(stream);

  if (dtype == PA_DTYPE_BF16 && varlen_tc_supported(head_dim, G, block_size) && max_query_len > 0) {
    // With a workspace, the short requests of the batch (decodes, verify blocks of up to
    // kShortRequestQueries queries) go to the split-KV decode, whose splits keep long contexts
    // streaming at HBM speed; a 128-row tensor-core tile would carry only their few rows, in one
    // CTA per request and KV head. The tensor-core kernel takes every other request, on a grid
    // planned on the device (only the tile pairs the batch has, longest first) unless the caller
    // passes a host plan. Launch order: the plan, the tensor-core grid, then the split-KV decode
    // as a programmatic dependent whose CTAs fill the SMs the tensor-core grid's tail leaves
    // free, and its combine.
    // a host plan: the short requests are on the split path iff there is a workspace (the plan
    // was made with the matching skip); otherwise the schedule decides, and a workspace carries
    // the device-planned work list
    if (workspace == nullptr && short_requests == PA_SHORT_SPLIT && work_items == nullptr)
      return PA_ERR_WORKSPACE_TOO_SMALL;
    const bool split_decodes =
        work_items != nullptr
            ? workspace != nullptr
            : workspace != nullptr &&
                  (short_requests == PA_SHORT_SPLIT ||
                   (short_requests == PA_SHORT_AUTO && num_reqs >= kAutoSplitMinReqs &&
                    (long long)num_tokens <= (long long)kAutoSplitMaxAvgQueries * num_reqs));
    const int skip_upto = split_decodes ? kShortRequestQueries : 0;
    const int q_tiles = (int)cdivll(max_query_len, varlen_tc_tokens_per_cta(G));
    int32_t* plan_items = nullptr;
    int plan_capacity = 0;
    if (workspace != nullptr && work_items == nullptr) {
      const long long cap = varlen_device_plan_capacity(num_reqs, num_tokens, max_query_len, G, skip_upto);
      const size_t plan_bytes = varlen_plan_bytes(num_reqs, max_query_len);
      if ((size_t)cap * 4 > plan_bytes || workspace_bytes < plan_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
      if (!aligned16(workspace)) return PA_ERR_INVALID_ARGUMENT;
      plan_items = static_cast<int32_t*>(workspace);
      plan_capacity = (int)cap;
      workspace = static_cast<uint8_t*>(workspace) + plan_bytes;
      workspace_bytes -= plan_bytes;
    }
    VarlenParams vp{};
    vp.skip_upto = skip_upto;
    vp.query_start_loc = query_start_loc;
    vp.seq_lens = seq_lens;
    vp.block_tables = block_tables;
    vp.out = out;
    vp.err = error_word;
    vp.num_reqs = num_reqs;
    vp.num_tokens = num_tokens;
    vp.num_q_heads = num_q_heads;
    vp.num_kv_heads = num_kv_heads;
    vp.group = G;
    vp.head_dim = head_dim;
    vp.block_size = block_size;
    vp.num_blocks = num_blocks;
    vp.max_blocks = max_blocks_per_seq;
    vp.max_query_len = max_query_len;
    vp.out_stride = out_stride;
    if (plan_items != nullptr) {
      vp.work_items = plan_items;
      vp.num_items = plan_capacity;
      vp.plan_on_device = 1;
    } else {
      vp.work_items = work_items;
      vp.num_items = work_items != nullptr ? num_items : 0;
    }
    const int tokens_per_tile = 128 / G;
    vp.q_tiles = q_tiles;
    vp.causal = causal ? 1 : 0;
    vp.scale_log2 = sc * kLog2e;
    st = apply_options(options, sc, vp);
    if (st != PA_OK) return st;
    CUtensorMap qmap, kmap, vmap;
    if (!encode_query_map(&qmap, q, head_dim, num_q_heads, num_tokens, G, tokens_per_tile, q_stride) ||
        !encode_varlen_cache_map(&kmap, k_cache, head_dim, num_kv_heads, block_size, num_blocks) ||
        !encode_varlen_cache_map(&vmap, v_cache, head_dim, num_kv_heads, block_size, num_blocks))
      return PA_ERR_CUDA;
    DecodeParams dp{};
    if (split_decodes) {
      dp.q = q;
      dp.k_cache = k_cache;
      dp.v_cache = v_cache;
      dp.block_tables = block_tables;
      dp.query_start_loc = query_start_loc;
      dp.seq_lens = seq_lens;
      dp.out = out;
      dp.err = error_word;
      dp.varlen = 2;
      dp.causal = causal ? 1 : 0;
      dp.num_reqs = num_reqs;
      dp.unit_tokens = short_unit_tokens(G);
      dp.groups_per_req = (int)cdivll(kShortRequestQueries, dp.unit_tokens);
      dp.small_max = kShortRequestQueries;
      dp.num_tokens = num_tokens;
      if ((long long)num_reqs * dp.groups_per_req * num_kv_heads * kShortRequestMaxSplits > (1ll << 31) - 1)
        return PA_ERR_UNSUPPORTED;
      dp.num_units = num_reqs * dp.groups_per_req;
      dp.num_q_heads = num_q_heads;
      dp.num_kv_heads = num_kv_heads;
      dp.group = G;
      dp.head_dim = head_dim;
      dp.block_size = block_size;
      dp.num_blocks = num_blocks;
      dp.max_blocks = max_blocks_per_seq;
      dp.q_stride = q_stride;
      dp.out_stride = out_stride;
      dp.scale_log2 = sc * kLog2e;
      dp.overlap_previous = 1;
      st = apply_options(options, sc, dp);
      if (st != PA_OK) return st;
      st = check_decode_units_workspace(dp, workspace, workspace_bytes);
      if (st != PA_OK) return st;
    }
    if (plan_items != nullptr &&
        launch_varlen_device_plan(query_start_loc, seq_lens, num_reqs, num_tokens, G, q_tiles, causal ? 1 : 0,
                                  vp.window, skip_upto, plan_items, plan_capacity, error_word, s) != cudaSuccess)
      return PA_ERR_CUDA;
    if (launch_varlen_tc(vp, qmap, kmap, vmap, s) != cudaSuccess) return PA_ERR_CUDA;
    if (split_decodes) return run_decode_units(dp, PA_DTYPE_BF16, k_cache, v_cache, 0, workspace, workspace_bytes, s);
    return PA_OK;
  }

  // Generic path: every query token is a decode over the keys it sees (one split).
  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.err = error_word;
  p.varlen = 1;
  p.causal = causal ? 1 : 0;
  p.num_reqs = num_reqs;
  p.num_units = num_tokens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = G;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.q_stride = q_stride;
  p.out_stride = out_stride;
  p.scale_log2 = sc * kLog2e;
  st = apply_options(options, sc, p);
  if (st != PA_OK) return st;
  return run_decode_units(p, dtype, k_cache, v_cache, 1, nullptr, 0, s);
}
}  // namespace
}  // namespace pa

extern "C" pa_status pa_paged_attention_varlen_planned(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* block_tables, int num_reqs, int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int causal, float scale, pa_dtype dtype,
    void* out, const pa_attn_options* options, const pa_row_strides* strides, void* workspace, size_t workspace_bytes,
    const int32_t* work_items, int num_items, int32_t* error_word, void* stream) {
  return varlen_impl(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs, num_tokens,
                     max_query_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                     causal, scale, dtype, out, options, strides, PA_SHORT_AUTO, workspace, workspace_bytes,
                     work_items, num_items, error_word, stream);
}

extern "C" pa_status pa_paged_attention_varlen_sched(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* block_tables, int num_reqs, int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, int max_blocks_per_seq, int causal, float scale, pa_dtype dtype,
    void* out, const pa_attn_options* options, const pa_row_strides* strides, pa_short_requests short_requests,
    void* workspace, size_t workspace_bytes, int32_t* error_word, void* stream) {
  return varlen_impl(q, k_cache, v_cache, query_start_loc, seq_lens, block_tables, num_reqs, num_tokens,
                     max_query_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq,
                     causal, scale, dtype, out, options, strides, (int)short_requests, workspace, workspace_bytes,
                     nullptr, 0, error_word, stream);
}

// ------------------------------------------------------------------------------ 8-bit caches
namespace {

int quant_kind(pa_dtype cache_dtype) {
  return cache_dtype == PA_DTYPE_INT8 ? 1 : (cache_dtype == PA_DTYPE_FP8_E4M3 ? 2 : 0);
}

// Shapes the 8-bit paths serve: bf16 queries, D 128 or 256 (a cached row spans whole 128-byte
// columns), groups up to 16, 16-token chunks.
pa_status validate_quant(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                         const float* v_scales, pa_dtype cache_dtype, const int32_t* block_tables, const void* out,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         int max_blocks_per_seq, float scale) {
  if (!k_scales || !v_scales) return PA_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(k_scales) & 3u) || (reinterpret_cast<uintptr_t>(v_scales) & 3u))
    return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_common(q, k_cache, v_cache, block_tables, out, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, scale, PA_DTYPE_BF16);
  if (st != PA_OK) return st;
  if (quant_kind(cache_dtype) == 0) return PA_ERR_UNSUPPORTED;
  if (head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_reshape_and_cache_quant(const void* key, const void* value, pa_dtype src_dtype,
                                                void* k_cache, void* v_cache, float* k_scales, float* v_scales,
                                                pa_dtype cache_dtype, const int32_t* slot_mapping, int num_tokens,
                                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                                int32_t* error_word, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (src_dtype != PA_DTYPE_BF16 && src_dtype != PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
  if (quant_kind(cache_dtype) == 0) return PA_ERR_UNSUPPORTED;
  if (head_dim % 32 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scales || !v_scales || !slot_mapping)
    return PA_ERR_INVALID_ARGUMENT;
  cudaError_t e = launch_reshape_and_cache_quant(key, value, src_dtype == PA_DTYPE_BF16, k_cache, v_cache, k_scales,
                                                 v_scales, cache_dtype == PA_DTYPE_FP8_E4M3, slot_mapping, num_tokens,
                                                 num_kv_heads, head_dim, (long long)num_blocks * block_size,
                                                 error_word, as_stream(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_paged_attention_decode_quant(const void* q, const void* k_cache, const void* v_cache,
                                                     const float* k_scales, const float* v_scales,
                                                     pa_dtype cache_dtype, const int32_t* block_tables,
                                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                                     int max_blocks_per_seq, float scale, int num_splits, void* out,
                                                     void* workspace, size_t workspace_bytes,
                                                     const pa_attn_options* options, int32_t* error_word,
                                                     void* stream) {
  if (num_seqs < 0 || num_splits < 0 || num_splits > kMaxSplits) return PA_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PA_OK;
  if (!context_lens) return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_quant(q, k_cache, v_cache, k_scales, v_scales, cache_dtype, block_tables, out, num_q_heads,
                                num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale);
  if (st != PA_OK) return st;
  if ((long long)num_seqs * num_kv_heads * kMaxSplits > (1ll << 31) - 1) return PA_ERR_UNSUPPORTED;
  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = error_word;
  p.num_units = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.quant = quant_kind(cache_dtype);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  const float sc = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;
  p.scale_log2 = sc * kLog2e;
  st = apply_options(options, sc, p);
  if (st != PA_OK) return st;
  if (num_splits == 0 && decode_seg_supported(head_dim, p.group, num_seqs, p.quant)) {
    // automatic splitting: balanced segments, every CTA that fits at once taking the same share of
    // the batch's chunks (with one split per sequence the 8-bit decode's last wave runs part full)
    DeviceInfo* info = nullptr;
    if (!device_info(&info)) return PA_ERR_CUDA;
    const int X = std::max(1, info->sms * decode_seg_ctas_per_sm(p.quant) / num_kv_heads);
    const size_t need = decode_seg_workspace_bytes(num_seqs, num_q_heads, X);
    if (workspace != nullptr && workspace_bytes >= need && aligned16(workspace)) {
      p.seg_ctas = X;
      p.ws_acc = static_cast<float*>(workspace);
      p.ws_ml = p.ws_acc + (size_t)X * 2 * num_q_heads * head_dim;
      p.seg_off = reinterpret_cast<int32_t*>(p.ws_ml + (size_t)X * 2 * num_q_heads * 2);
      p.q_stride = (long long)num_q_heads * head_dim;
      p.out_stride = (long long)num_q_heads * head_dim;
      CUtensorMap kmap, vmap;
      if (!encode_cache_map(&kmap, k_cache, head_dim, num_kv_heads, block_size, num_blocks, kChunk, 1) ||
          !encode_cache_map(&vmap, v_cache, head_dim, num_kv_heads, block_size, num_blocks, kChunk, 1))
        return PA_ERR_CUDA;
      return launch_decode_seg(p, kmap, vmap, as_stream(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
  }
  return run_decode_units(p, PA_DTYPE_BF16, k_cache, v_cache, num_splits, workspace, workspace_bytes,
                          as_stream(stream));
}

extern "C" pa_status pa_paged_attention_varlen_quant(const void* q, const void* k_cache, const void* v_cache,
                                                     const float* k_scales, const float* v_scales,
                                                     pa_dtype cache_dtype, const int32_t* query_start_loc,
                                                     const int32_t* seq_lens, const int32_t* block_tables,
                                                     int num_reqs, int num_tokens, int max_query_len,
                                                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                                     int num_blocks, int max_blocks_per_seq, int causal, float scale,
                                                     void* out, const pa_attn_options* options, int32_t* error_word,
                                                     void* stream) {
  if (num_reqs < 0 || num_tokens < 0 || max_query_len < 0) return PA_ERR_INVALID_ARGUMENT;
  if (num_reqs == 0 || num_tokens == 0) return PA_OK;
  if (!query_start_loc || !seq_lens) return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_quant(q, k_cache, v_cache, k_scales, v_scales, cache_dtype, block_tables, out, num_q_heads,
                                num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale);
  if (st != PA_OK) return st;
  if ((long long)num_tokens * num_kv_heads > (1ll << 31) - 1) return PA_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  const float sc = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;
  if (head_dim == 128 && varlen_tc_supported(head_dim, G, block_size) && max_query_len > 0) {
    // the tensor-core kernel: each K / V tile's codes are dequantised to bf16 in shared memory
    // ("32. Production attention kernels", Quantized KV caches), then used like a bf16 tile
    VarlenParams vp{};
    vp.query_start_loc = query_start_loc;
    vp.seq_lens = seq_lens;
    vp.block_tables = block_tables;
    vp.out = out;
    vp.err = error_word;
    vp.num_reqs = num_reqs;
    vp.num_tokens = num_tokens;
    vp.num_q_heads = num_q_heads;
    vp.num_kv_heads = num_kv_heads;
    vp.group = G;
    vp.head_dim = head_dim;
    vp.block_size = block_size;
    vp.num_blocks = num_blocks;
    vp.max_blocks = max_blocks_per_seq;
    vp.max_query_len = max_query_len;
    vp.q_tiles = (int)cdivll(max_query_len, varlen_tc_tokens_per_cta(G));
    vp.causal = causal ? 1 : 0;
    vp.scale_log2 = sc * kLog2e;
    vp.quant = quant_kind(cache_dtype);
    vp.k_scales = k_scales;
    vp.v_scales = v_scales;
    st = apply_options(options, sc, vp);
    if (st != PA_OK) return st;
    CUtensorMap qmap, kmap, vmap;
    const int box = block_size < 128 ? block_size : 128;
    if (!encode_query_map(&qmap, q, head_dim, num_q_heads, num_tokens, G, 128 / G,
                          (long long)num_q_heads * head_dim) ||
        !encode_cache_map(&kmap, k_cache, head_dim, num_kv_heads, block_size, num_blocks, box, 1) ||
        !encode_cache_map(&vmap, v_cache, head_dim, num_kv_heads, block_size, num_blocks, box, 1))
      return PA_ERR_CUDA;
    return launch_varlen_tc(vp, qmap, kmap, vmap, as_stream(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.err = error_word;
  p.varlen = 1;
  p.causal = causal ? 1 : 0;
  p.num_reqs = num_reqs;
  p.num_units = num_tokens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.quant = quant_kind(cache_dtype);
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.scale_log2 = sc * kLog2e;
  st = apply_options(options, sc, p);
  if (st != PA_OK) return st;
  return run_decode_units(p, PA_DTYPE_BF16, k_cache, v_cache, 1, nullptr, 0, as_stream(stream));
}

extern "C" pa_status pa_selftest_wait_timeout(int limit_us, int32_t* error_word, void* stream) {
  if (limit_us < 1 || limit_us > 1000000 || error_word == nullptr) return PA_ERR_INVALID_ARGUMENT;
  return launch_wait_timeout_selftest((uint64_t)limit_us * 1000ull, error_word, as_stream(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// ------------------------------------------------------------------------------ cascade
namespace {

// The combine merges at most kMaxSplits partials per row: up to kMaxPrefixSplits key ranges
// of the prefix, the rest for the suffix's splits.
constexpr int kMaxPrefixSplits = 16;
constexpr int kMinPrefixTilesPerSplit = 2;  // 256 keys: keeps the Q load and pipeline fill amortised

struct CascadePlan {
  int prefix_splits, prefix_per;  // key ranges of the prefix pass, 128-key tiles each
  int suffix_splits, suffix_per;  // splits of the suffix decode, 16-key chunks each
};

long long prefix_tiles_bound(int max_prefix_blocks, int block_size) {
  return cdivll((long long)max_prefix_blocks * block_size, 128);
}

// Prefix ranges fill the SMs for the q_tiles x Hkv tiles of the pass (the prefix length itself
// is a device value: ranges past its end write neutral partials); the suffix gets the splits
// the plain decode would pick, within what is left of the combine's budget.
CascadePlan cascade_plan(DeviceInfo* info, int num_seqs, int Hkv, int D, int G, int block_size,
                         int max_prefix_blocks, int max_blocks_per_seq, int num_splits) {
  CascadePlan c;
  const long long ptiles = prefix_tiles_bound(max_prefix_blocks, block_size);
  const long long base_ctas = cdivll(num_seqs, varlen_tc_tokens_per_cta(G)) * Hkv;
  long long ps = cdivll(info->sms, base_ctas);
  ps = std::min<long long>(ps, std::min<long long>(kMaxPrefixSplits, cdivll(ptiles, kMinPrefixTilesPerSplit)));
  ps = std::max<long long>(ps, 1);
  c.prefix_per = (int)cdivll(ptiles, ps);
  c.prefix_splits = (int)cdivll(ptiles, c.prefix_per);
  const long long max_chunks = cdivll((long long)max_blocks_per_seq * block_size, kChunk);
  int ss = num_splits > 0 ? num_splits : auto_splits(info, num_seqs, Hkv, D, G, max_chunks, PA_DTYPE_BF16);
  ss = (int)std::min<long long>(std::min(ss, kMaxSplits - c.prefix_splits), max_chunks);
  c.suffix_per = (int)cdivll(max_chunks, ss);
  c.suffix_splits = (int)cdivll(max_chunks, c.suffix_per);
  return c;
}

}  // namespace

extern "C" size_t pa_cascade_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int block_size,
                                             int max_prefix_blocks, int max_blocks_per_seq) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_prefix_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const long long ptiles = prefix_tiles_bound(max_prefix_blocks, block_size);
  const long long ps = std::min<long long>(kMaxPrefixSplits, cdivll(ptiles, kMinPrefixTilesPerSplit));
  const long long max_chunks = cdivll((long long)max_blocks_per_seq * block_size, kChunk);
  const long long slots = std::min<long long>(kMaxSplits, ps + max_chunks);
  return (size_t)((long long)num_seqs * slots * num_q_heads * ((long long)head_dim + 2) * 4);
}

extern "C" pa_status pa_cascade_decode(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* prefix_table, const int32_t* prefix_len, int max_prefix_blocks,
                                       const int32_t* suffix_tables, const int32_t* suffix_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, int max_blocks_per_seq, float scale, int num_splits, void* out,
                                       void* workspace, size_t workspace_bytes, int32_t* error_word, void* stream) {
  if (num_seqs < 0 || num_splits < 0 || num_splits > kMaxSplits - 1 || max_prefix_blocks <= 0)
    return PA_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0) return PA_OK;
  if (!prefix_table || !prefix_len || !suffix_lens) return PA_ERR_INVALID_ARGUMENT;
  pa_status st = validate_common(q, k_cache, v_cache, suffix_tables, out, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks_per_seq, scale, PA_DTYPE_BF16);
  if (st != PA_OK) return st;
  const int G = num_q_heads / num_kv_heads;
  if (!varlen_tc_prefix_supported(head_dim, G, block_size)) return PA_ERR_UNSUPPORTED;
  if ((long long)max_prefix_blocks * block_size > (1ll << 30)) return PA_ERR_UNSUPPORTED;
  if ((long long)num_seqs * num_kv_heads * kMaxSplits > (1ll << 31) - 1) return PA_ERR_UNSUPPORTED;
  DeviceInfo* info = nullptr;
  if (!device_info(&info)) return PA_ERR_CUDA;
  cudaStream_t strm = as_stream(stream);
  const float sc = scale == 0.f ? 1.f / sqrtf((float)head_dim) : scale;

  const CascadePlan plan = cascade_plan(info, num_seqs, num_kv_heads, head_dim, G, block_size, max_prefix_blocks,
                                        max_blocks_per_seq, num_splits);
  const int slots = plan.prefix_splits + plan.suffix_splits;
  const size_t need = (size_t)num_seqs * slots * num_q_heads * ((size_t)head_dim + 2) * 4;
  if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return PA_ERR_INVALID_ARGUMENT;
  float* ws_acc = static_cast<float*>(workspace);
  float* ws_ml = ws_acc + (size_t)num_seqs * slots * num_q_heads * head_dim;

  // 1. the shared prefix, read once per key range: all S * G query rows of a KV head against
  //    its pages, partials to slots [0, prefix_splits)
  VarlenParams vp{};
  vp.block_tables = prefix_table;
  vp.out = out;
  vp.err = error_word;
  vp.num_reqs = plan.prefix_splits;
  vp.num_tokens = num_seqs;
  vp.num_q_heads = num_q_heads;
  vp.num_kv_heads = num_kv_heads;
  vp.group = G;
  vp.head_dim = head_dim;
  vp.block_size = block_size;
  vp.num_blocks = num_blocks;
  vp.max_blocks = max_prefix_blocks;
  vp.max_query_len = num_seqs;
  vp.q_tiles = (int)cdivll(num_seqs, varlen_tc_tokens_per_cta(G));
  vp.causal = 0;
  vp.scale_log2 = sc * kLog2e;
  vp.prefix_mode = 1;
  vp.prefix_len = prefix_len;
  vp.prefix_tiles_per_split = plan.prefix_per;
  vp.ws_acc = ws_acc;
  vp.ws_ml = ws_ml;
  vp.slot_count = slots;
  CUtensorMap qmap, kmap, vmap;
  if (!encode_query_map(&qmap, q, head_dim, num_q_heads, num_seqs, G, 128 / G, (long long)num_q_heads * head_dim) ||
      !encode_varlen_cache_map(&kmap, k_cache, head_dim, num_kv_heads, block_size, num_blocks) ||
      !encode_varlen_cache_map(&vmap, v_cache, head_dim, num_kv_heads, block_size, num_blocks))
    return PA_ERR_CUDA;
  if (launch_varlen_tc(vp, qmap, kmap, vmap, strm) != cudaSuccess) return PA_ERR_CUDA;

  // 2. each sequence's own suffix: the split-KV decode, partials to the slots after the prefix's
  DecodeParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = suffix_tables;
  p.context_lens = suffix_lens;
  p.out = out;
  p.err = error_word;
  p.num_units = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = G;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_blocks = max_blocks_per_seq;
  p.scale_log2 = sc * kLog2e;
  p.num_splits = plan.suffix_splits;
  p.chunks_per_split = plan.suffix_per;
  p.ws_acc = ws_acc;
  p.ws_ml = ws_ml;
  p.force_partial = 1;
  p.slot_offset = plan.prefix_splits;
  p.slot_count = slots;
  // the suffixes read nothing the prefix pass writes: their CTAs may start on the SMs the prefix
  // pass leaves free, while it runs (they finish only after it, for the combine's sake)
  p.overlap_previous = 1;
  CUtensorMap skmap, svmap;
  if (!encode_decode_cache_map(&skmap, k_cache, head_dim, num_kv_heads, block_size, num_blocks, kChunk) ||
      !encode_decode_cache_map(&svmap, v_cache, head_dim, num_kv_heads, block_size, num_blocks, kChunk))
    return PA_ERR_CUDA;
  if (launch_decode_bf16(p, skmap, svmap, strm) != cudaSuccess) return PA_ERR_CUDA;

  // 3. merge every row's prefix and suffix partials (the split-KV combine over all its slots)
  DecodeParams c = p;
  c.num_splits = slots;
  return launch_combine(c, PA_DTYPE_BF16, strm) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
