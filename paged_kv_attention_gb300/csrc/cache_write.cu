// reshape_and_cache: scatter this step's key/value rows into the paged pools.
//
// For token i with slot = slot_mapping[i] >= 0, the Hkv*D elements of key[i] go to
// k_cache[slot / block_size, slot % block_size] (and value[i] to v_cache): in the
// [num_blocks, block_size, Hkv, D] layout that destination row is contiguous, so slot s
// simply starts at element s * Hkv * D. A bit-exact copy; -1 writes nothing.
// ("poot - Attention and KV Cache", KV cache: the write map; "32. Production attention
// kernels", Quantized KV caches: write_kv through meta.slot_mapping.)
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// One warp per token; 16-byte vector copies (every row is a multiple of 16 bytes).
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ key,
                                                                const uint4* __restrict__ value,
                                                                uint4* __restrict__ k_cache,
                                                                uint4* __restrict__ v_cache,
                                                                const int32_t* __restrict__ slot_mapping,
                                                                int num_tokens, int row_vecs, long long num_slots,
                                                                int32_t* err) {
  const int token = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int slot = slot_mapping[token];
  if (slot < 0 || (long long)slot >= num_slots) {
    if (slot != -1 && lane == 0) flag_error(err, PA_ERRBIT_SLOT_OUT_OF_POOL);
    return;
  }
  const uint4* ks = key + (size_t)token * row_vecs;
  const uint4* vs = value + (size_t)token * row_vecs;
  uint4* kd = k_cache + (size_t)slot * row_vecs;
  uint4* vd = v_cache + (size_t)slot * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) {
    const uint4 a = __ldg(ks + i);
    const uint4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int32_t* slot_mapping, int num_tokens, int row_bytes,
                                     long long num_slots, int32_t* err, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((num_tokens + 7) / 8);
  reshape_and_cache_kernel<<<blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, num_tokens, row_bytes / 16, num_slots, err);
  return cudaGetLastError();
}

}  // namespace pa
