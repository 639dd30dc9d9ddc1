// reshape_and_cache: scatter this step's key/value rows into the paged pools.
//
// For token i with slot = slot_mapping[i] >= 0, the Hkv*D elements of key row i go to
// k_cache[slot / block_size, slot % block_size] (and value[i] to v_cache): in the
// [num_blocks, block_size, Hkv, D] layout that destination row is contiguous, so slot s
// simply starts at element s * Hkv * D. A bit-exact copy; -1 writes nothing.
// ("poot - Attention and KV Cache", KV cache: the write map; "32. Production attention
// kernels", Quantized KV caches: write_kv through meta.slot_mapping.)
#include <cuda_fp8.h>

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
                                                                int num_tokens, int row_vecs, long long key_vecs,
                                                                long long value_vecs, long long num_slots,
                                                                int32_t* err) {
  const int token = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int slot = slot_mapping[token];
  if (slot < 0 || (long long)slot >= num_slots) {
    if (slot != -1 && lane == 0) flag_error(err, PA_ERRBIT_SLOT_OUT_OF_POOL);
    return;
  }
  const uint4* ks = key + (size_t)token * key_vecs;
  const uint4* vs = value + (size_t)token * value_vecs;
  uint4* kd = k_cache + (size_t)slot * row_vecs;
  uint4* vd = v_cache + (size_t)slot * row_vecs;
  for (int i = lane; i < row_vecs; i += 32) {
    const uint4 a = __ldg(ks + i);
    const uint4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

// Quantising write: one warp per (token, KV head); lane l holds elements l, l+32, ... of the
// head's row. Float32 throughout, IEEE divisions, round half to even: the same operations,
// in the same precision, as the page's quantiser, so codes and scales are reproducible.
template <typename SrcT, int KIND>  // KIND 0: int8 (q_max 127), 1: fp8 E4M3 (q_max 448)
__global__ void __launch_bounds__(256) reshape_and_cache_quant_kernel(
    const SrcT* __restrict__ key, const SrcT* __restrict__ value, uint8_t* __restrict__ k_cache,
    uint8_t* __restrict__ v_cache, float* __restrict__ k_scales, float* __restrict__ v_scales,
    const int32_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads, int head_dim, long long num_slots,
    int32_t* err) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)num_tokens * num_kv_heads) return;
  const int token = (int)(wid / num_kv_heads);
  const int h = (int)(wid - (long long)token * num_kv_heads);
  const int slot = slot_mapping[token];
  if (slot < 0 || (long long)slot >= num_slots) {
    if (slot != -1 && lane == 0 && h == 0) flag_error(err, PA_ERRBIT_SLOT_OUT_OF_POOL);
    return;
  }
  constexpr float kQMax = KIND == 0 ? 127.f : 448.f;
  const size_t src = ((size_t)token * num_kv_heads + h) * head_dim;
  const size_t dst = ((size_t)slot * num_kv_heads + h) * head_dim;
  for (int which = 0; which < 2; ++which) {
    const SrcT* x = (which == 0 ? key : value) + src;
    uint8_t* codes = (which == 0 ? k_cache : v_cache) + dst;
    float amax = 0.f;
    for (int d = lane; d < head_dim; d += 32) amax = fmaxf(amax, fabsf(static_cast<float>(x[d])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    amax = fmaxf(amax, 1e-8f);
    const float scale = __fdiv_rn(amax, kQMax);
    for (int d = lane; d < head_dim; d += 32) {
      const float y = __fdiv_rn(static_cast<float>(x[d]), scale);
      uint8_t c;
      if (KIND == 0) {
        const float r = fminf(fmaxf(rintf(y), -127.f), 127.f);
        c = static_cast<uint8_t>(static_cast<int8_t>(r));
      } else {
        c = static_cast<uint8_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
      }
      codes[d] = c;
    }
    if (lane == 0) ((which == 0 ? k_scales : v_scales))[(size_t)slot * num_kv_heads + h] = scale;
  }
}

// Self-test of the bounded wait every pipelined kernel uses: one thread waits on a fresh
// mbarrier that nothing will ever arrive at, with the given limit, and reports the expiry
// through the error word exactly as a kernel does. No other thread waits on anything.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait(&bar, 0, limit_ns)) flag_error(err, PA_ERRBIT_WAIT_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int32_t* err, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_quant(const void* key, const void* value, bool src_bf16, void* k_cache,
                                           void* v_cache, float* k_scales, float* v_scales, bool fp8,
                                           const int32_t* slot_mapping, int num_tokens, int num_kv_heads,
                                           int head_dim, long long num_slots, int32_t* err, cudaStream_t stream) {
  const long long warps = (long long)num_tokens * num_kv_heads;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
#define PA_QW(T, K)                                                                                          \
  reshape_and_cache_quant_kernel<T, K><<<blocks, 256, 0, stream>>>(                                          \
      static_cast<const T*>(key), static_cast<const T*>(value), kc, vc, k_scales, v_scales, slot_mapping,    \
      num_tokens, num_kv_heads, head_dim, num_slots, err)
  if (src_bf16) {
    if (fp8) PA_QW(__nv_bfloat16, 1); else PA_QW(__nv_bfloat16, 0);
  } else {
    if (fp8) PA_QW(float, 1); else PA_QW(float, 0);
  }
#undef PA_QW
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int32_t* slot_mapping, int num_tokens, int row_bytes,
                                     long long key_stride, long long value_stride, long long num_slots,
                                     int32_t* err, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((num_tokens + 7) / 8);
  reshape_and_cache_kernel<<<blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, num_tokens, row_bytes / 16, key_stride / 16, value_stride / 16,
      num_slots, err);
  return cudaGetLastError();
}

}  // namespace pa
