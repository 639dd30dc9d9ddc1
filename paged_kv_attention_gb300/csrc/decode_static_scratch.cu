// pa_paged_attention_decode_static_scratch: the split-KV decode for callers that cannot
// allocate device memory.
//
// The regular decode entry point asks its caller for a workspace that holds the per-split
// partial results. Some callers have no way to provide one: a plugin that a host framework
// hands only its input and output pointers, with no allocator and no workspace hook; a
// runtime that carved all device memory into its own pools at start-up and forbids further
// cudaMalloc calls; or a latency-critical loop that cannot afford cudaMalloc's implicit
// device synchronisation. This entry point serves them from a fixed scratch array that lives
// in the library's own device image, so the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds its
// kStaticScratchBytes for the life of the process. Its address is looked up once per device
// with cudaGetSymbolAddress (on the first call made while that device is current).
#include <atomic>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace {

// 16 MiB: enough for the split partials of, for example, 64 sequences x 32 query heads x
// head_dim 128 at up to 15 splits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;

}  // namespace

// Device-side scratch shared by every call on a device. Host code must not use this name as
// a pointer (on the host it is only a stand-in); it uses the address that
// cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char pa_decode_static_scratch[kStaticScratchBytes];

namespace {

// Device address of the scratch array on the current device, looked up once per device and
// kept for the life of the process. After the first lookup a call reads the cached address
// with one acquire load; only a device's first lookup takes the lock. The cache is not
// refreshed after a device reset (cudaDeviceReset, or the primary context being released and
// re-created): the library does not support calling this entry point across one.
pa_status static_scratch_address(void** out) {
  static std::mutex mu;
  static std::atomic<void*> addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(mu);
    p = addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, pa_decode_static_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
      addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_paged_attention_decode_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, int max_blocks_per_seq, float scale, pa_dtype dtype, int num_splits, void* out,
    int32_t* error_word, void* stream) {
  void* scratch = nullptr;
  const pa_status st = static_scratch_address(&scratch);
  if (st != PA_OK) return st;
  // The regular entry point checks the partials' size against the array and refuses a batch
  // that does not fit (PA_ERR_WORKSPACE_TOO_SMALL) before anything is launched.
  return pa_paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                   num_kv_heads, head_dim, block_size, num_blocks, max_blocks_per_seq, scale, dtype,
                                   num_splits, out, scratch, kStaticScratchBytes, error_word, stream);
}
