// Varlen causal paged attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method ("32. Production attention kernels", One kernel for the whole batch;
// "TileInfer.jl - Attention kernels", Prefill and Walking the block table):
//  * a query tile is 128 packed rows: 128/G consecutive query tokens of one request times
//    the G query heads of one KV head (row m = token m / G, head m % G), so every K/V tile
//    serves the whole group;
//  * request r's q_len queries are the newest of its seq_len positions (query t sits at
//    seq_len - q_len + t) and see keys up to their own position; the key loop stops at the
//    tile's last query and only tiles that cross the diagonal or the sequence end are masked;
//  * FlashAttention-2 online softmax in fp32 with exp2 (scale pre-multiplied by log2 e);
//    probabilities are rounded to bf16 for the P.V product.
//
// GB300 mapping. One CTA owns two consecutive query tiles (A, B) of one (request, KV head)
// and streams the K/V tiles they need once for both:
//  * warp 8 (one lane) walks the block table and issues TMA loads: both Q tiles once, then
//    two-stage rings for K and V (128-key tiles, one box per page per 64-column half,
//    128-byte swizzle, the layout the tensor core reads directly);
//  * warp 9 owns the tensor memory (512 columns: S_A, S_B, O_A, O_B, 128 each) and one lane
//    issues tcgen05.mma (S: M=128 N=128 K=128 from shared memory; P.V: M=128 N=128 K=128
//    with A from TMEM) in the order S_A(j), S_B(j), PV_A(j), S_A(j+1), PV_B(j), S_B(j+1),
//    ... so that the tensor core works on one tile while the other tile's softmax runs;
//  * warps 0-3 (tile A) and 4-7 (tile B), one thread per row, read S from TMEM, mask, update
//    the running max/sum, write P as bf16 back into the first 64 columns of their S block
//    and signal; P.V then takes its A operand from TMEM (no shared-memory round trip for P).
//    O is rescaled in TMEM only when the running max rose by more than 2^8 (exact for any
//    reference max; this only bounds the range of P and O);
//  * every wait is bounded; on expiry the CTA flags PA_ERRBIT_WAIT_TIMEOUT, drains its
//    outstanding copies and MMAs, frees its tensor memory and exits.
#include <cuda_fp16.h>

#include <atomic>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kBM = 128;  // packed query rows per tile
constexpr int kStages = 2;
constexpr int kRegion = 128 * 128;  // one [128 rows][64 bf16] swizzled 64-column block: 16 KiB
constexpr int kLoneStages = 3;  // a CTA whose second query tile is empty keeps three K/V stages
enum {
  B_Q = 0,
  B_KF = 1,   // +stage (3)
  B_VF = 4,   // +stage
  B_KE = 7,   // +stage
  B_VE = 10,  // +stage
  B_SF = 13,  // +tile (A, B); a lone tile: +score block
  B_PR = 15,  // +tile; a lone tile: +score block
  B_OD = 17,  // +tile
  B_FIN = 19,
  B_KR = 20,  // +stage: 8-bit caches, the K tile is dequantised to bf16 (64 converter arrivals)
  B_VR = 22,  // +stage: the same for V
  kNumBars = 24
};
// Shared-memory layout for head dim kD (64 or 128): a tile of 128 rows is kD / 64 column blocks.
// kQ (8-bit caches: 1 int8, 2 fp8 E4M3): a stage's codes land in its second column block and
// are dequantised in place; its 128 key and 128 value scales sit after the V ring.
// bf16 tiles (kQ 0): a lone tile's third K stage takes Q_B's place and its third V stage the
// region after the barriers.
template <int kD, int kQ = 0>
struct Layout {
  static constexpr int kTileBytes = (kD / 64) * kRegion;
  static constexpr int kOffQ = 0;  // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffScale = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffScale + (kQ != 0 ? kStages * 256 * 4 : 0);
  static constexpr int kOffV2 = (kOffBar + kNumBars * 8 + 32 + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = 1024 + (kQ == 0 ? kOffV2 + kTileBytes : kOffBar + kNumBars * 8 + 32);
  static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");
  // stage st of K / V (st < kStages: the rings; st == kStages: a lone tile's third stage)
  __device__ static constexpr int k_stage(int st) { return st < kStages ? kOffK + st * kTileBytes : kOffQ + kTileBytes; }
  __device__ static constexpr int v_stage(int st) { return st < kStages ? kOffV + st * kTileBytes : kOffV2; }
  // Inside a K / V tile: bf16 tiles at head dim 128 arrive one page per copy as [8-row group]
  // [column block][8 rows x 128 bytes] (kWide), the others as [column block][128 rows x 128
  // bytes]. kCB: from one 64-column block to the next; kSBO: from one 8-row group to the next.
  static constexpr bool kWide = kQ == 0 && kD == 128;
  static constexpr int kCB = kWide ? 1024 : kRegion;
  static constexpr int kSBO = kWide ? 1024 * (kD / 64) : 1024;
  __device__ static constexpr int at(int row, int cb) { return (row >> 3) * kSBO + cb * kCB + (row & 7) * 128; }
};
constexpr int kThreads = 320;
constexpr int kThreadsQ = 384;  // 8-bit caches: two more warps dequantise the K / V tiles
constexpr uint32_t kTmemCols = 512;
// TMEM columns of tile t's score block and output accumulator (kD columns)
__host__ __device__ constexpr uint32_t col_s(int t) { return t == 0 ? 0u : 128u; }
template <int kD>
__host__ __device__ constexpr uint32_t col_o(int t) { return t == 0 ? 256u : 256u + kD; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// ---------------------------------------------------------------- 8-bit cache tiles
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Four int8 codes (one word) times the row's scale -> two bf16 pairs (dims in byte order). A
// code c becomes exactly c as a float through the bits 0x4B0000xx (2^23 + the byte of c + 128)
// minus 2^23 + 128; the product with the fp32 scale is rounded once to fp32, then to bf16.
__device__ __forceinline__ void int8x4_to_bf16(uint32_t w, uint64_t s2, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint64_t bias = f2(-8388736.f, -8388736.f);
  float a0, a1, a2, a3;
  f2_split(f2_mul(f2_add(f2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)),
                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541))),
                         bias),
                  s2),
           a0, a1);
  f2_split(f2_mul(f2_add(f2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542)),
                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543))),
                         bias),
                  s2),
           a2, a3);
  lo = pack_bf16x2(a0, a1);
  hi = pack_bf16x2(a2, a3);
}
// Four E4M3 codes times the scale -> two bf16 pairs: each code pair through the exact E4M3 -> f16x2
// conversion, widened to fp32, multiplied (one rounding), rounded to bf16.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint64_t s2, uint32_t& lo, uint32_t& hi) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  float a0, a1, a2, a3;
  f2_split(f2_mul(f2(f01.x, f01.y), s2), a0, a1);
  f2_split(f2_mul(f2(f23.x, f23.y), s2), a2, a3);
  lo = pack_bf16x2(a0, a1);
  hi = pack_bf16x2(a2, a3);
}
// Dequantise key / value row `row` of a head_dim-128 tile in place: its 128 codes sit in column
// block 1 (one 128-byte swizzled row), the bf16 row takes both 64-column blocks. The whole code row
// is read before any of it is overwritten, and no other row is touched.
template <int kQ>
__device__ __forceinline__ void dequantize_row(uint8_t* tile, int row, float scale, bool valid) {
  const uint32_t sw = (uint32_t)(row & 7);
  uint4 cw[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) cw[u] = *reinterpret_cast<const uint4*>(tile + kRegion + row * 128 + ((u ^ sw) << 4));
  const uint64_t s2 = f2(scale, scale);
#pragma unroll
  for (int u = 0; u < 8; ++u) {  // codes 16u .. 16u+15 -> bf16 units 2(u%4), 2(u%4)+1 of block u/4
    uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
    if (valid) {
      if constexpr (kQ == 1) {
        int8x4_to_bf16(cw[u].x, s2, o0.x, o0.y);
        int8x4_to_bf16(cw[u].y, s2, o0.z, o0.w);
        int8x4_to_bf16(cw[u].z, s2, o1.x, o1.y);
        int8x4_to_bf16(cw[u].w, s2, o1.z, o1.w);
      } else {
        e4m3x4_to_bf16(cw[u].x, s2, o0.x, o0.y);
        e4m3x4_to_bf16(cw[u].y, s2, o0.z, o0.w);
        e4m3x4_to_bf16(cw[u].z, s2, o1.x, o1.y);
        e4m3x4_to_bf16(cw[u].w, s2, o1.z, o1.w);
      }
    }
    uint8_t* blk = tile + (u >> 2) * kRegion + row * 128;
    const uint32_t k0 = 2u * (uint32_t)(u & 3);
    *reinterpret_cast<uint4*>(blk + ((k0 ^ sw) << 4)) = o0;
    *reinterpret_cast<uint4*>(blk + (((k0 + 1) ^ sw) << 4)) = o1;
  }
}

// kPrefix: the cascade's shared-prefix pass (one request of num_tokens query rows that all
// see the whole prefix; unnormalised partials out instead of normalised rows).
template <bool kPrefix, int kD, int kQ = 0>
__global__ void __launch_bounds__(kQ != 0 ? kThreadsQ : kThreads, 1)
    varlen_tc_kernel(const __grid_constant__ VarlenParams p, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  static_assert(kQ == 0 || (kD == 128 && !kPrefix), "8-bit caches: head_dim 128, no prefix mode");
  constexpr int kTileBytes = Layout<kD, kQ>::kTileBytes;
  constexpr int kOffQ = Layout<kD, kQ>::kOffQ;
  constexpr int kOffK = Layout<kD, kQ>::kOffK;
  constexpr int kOffV = Layout<kD, kQ>::kOffV;
  constexpr int kOffScale = Layout<kD, kQ>::kOffScale;
  constexpr int kOffBar = Layout<kD, kQ>::kOffBar;
  constexpr int kBlocks = kD / 64;  // 64-column blocks of a row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_k = reinterpret_cast<int*>(tmem_slot + 2);  // K / V tiles whose copies are out
  int* issued_v = reinterpret_cast<int*>(tmem_slot + 3);

  // ---- which tile pair: from the caller's plan (heaviest first by the host's estimate, no empty
  // pairs), else heaviest (last) query tiles first across all requests and heads
  int tile, r, kvh;  // r: the request, or the prefix key range in prefix mode
  if (!kPrefix && p.work_items != nullptr) {
    // a list planned on the device by the kernel launched just before this one: wait for it
    if (p.plan_on_device) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int item = p.plan_on_device ? p.work_items[blockIdx.x / p.num_kv_heads]
                                      : __ldg(p.work_items + blockIdx.x / p.num_kv_heads);
    kvh = (int)(blockIdx.x % p.num_kv_heads);
    if (item < 0) return;  // padding past the plan's last item
    tile = item / p.num_reqs;
    r = item - tile * p.num_reqs;
    if (tile >= p.q_tiles) {  // not an item of this batch: nothing to do here
      if (threadIdx.x == 0 && kvh == 0) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
      return;
    }
  } else {
    // heaviest (last) query tiles first, in chunks of 16 tile indices; within a chunk the pairs of
    // one (request, KV head) are consecutive, so the CTAs running side by side read the same K/V
    // tiles at about the same time and mostly from L2 (bf16 at head dim 128; the other variants
    // measured faster in the plain order, chunks of one tile index)
    constexpr int kChunkTiles = (kQ == 0 && kD == 128 && !kPrefix) ? 16 : 1;
    const int per_tile = p.num_reqs * p.num_kv_heads;
    const long long chunk_span = (long long)kChunkTiles * per_tile;
    const int c = (int)(blockIdx.x / chunk_span);
    const int in_chunk = (int)(blockIdx.x % chunk_span);
    const int tiles_here = min(kChunkTiles, p.q_tiles - c * kChunkTiles);
    const int combo = in_chunk / tiles_here;
    tile = p.q_tiles - 1 - (c * kChunkTiles + in_chunk % tiles_here);
    r = combo / p.num_kv_heads;
    kvh = combo - r * p.num_kv_heads;
  }
  const int G = p.group;
  const int TOK = kBM / G;  // tokens per 128-row tile; a CTA covers 2 * TOK tokens
  const int tid = threadIdx.x;

  int q_start, q_stop, seq_len;
  if (kPrefix) {
    // the cascade's shared prefix: every query row attends to all of it
    q_start = 0;
    q_stop = p.num_tokens;
    seq_len = *p.prefix_len;
    const int cap = p.max_blocks * p.block_size;
    if (seq_len < 0 || seq_len > cap) {
      if (tid == 0 && kvh == 0 && tile == 0) flag_error(p.err, PA_ERRBIT_LENGTH_OUT_OF_RANGE);
      seq_len = seq_len < 0 ? 0 : cap;
    }
  } else {
    q_start = p.query_start_loc[r];
    q_stop = p.query_start_loc[r + 1];
    seq_len = p.seq_lens[r];
    // short requests (decodes, verify blocks) left to the split-KV decode launched beside it
    // (a malformed block, reaching past the last row, stays here to be flagged)
    if (q_start >= 0 && q_stop <= p.num_tokens && q_stop - q_start >= 1 && q_stop - q_start <= p.skip_upto) return;
  }
  const int q_len = q_stop - q_start;
  const bool layout_ok = q_start >= 0 && q_len >= 0 && q_stop <= p.num_tokens;
  const bool too_long = seq_len > p.max_blocks * p.block_size;
  const bool bad = !layout_ok || (!kPrefix && (q_len > seq_len || too_long));
  const int tok0 = tile * 2 * TOK;
  if (bad) {
    if (tid == 0 && kvh == 0 && tile == 0)
      flag_error(p.err, too_long && layout_ok && q_len <= seq_len ? PA_ERRBIT_LENGTH_OUT_OF_RANGE
                                                                   : PA_ERRBIT_QUERY_LAYOUT);
    if (!layout_ok || tok0 >= q_len) return;
    // a request the kernel cannot serve gives zero rows
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    const int rows = min(2 * TOK, q_len - tok0) * G;
    for (int i = tid; i < rows * (kD / 8); i += blockDim.x) {
      const int row = i / (kD / 8), c = i % (kD / 8);
      const size_t o = (size_t)(q_start + tok0 + row / G) * p.out_stride + (size_t)(kvh * G + row % G) * kD + c * 8;
      *reinterpret_cast<uint4*>(out + o) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  if (tile == 0 && kvh == 0 && tid == 0 && q_len > p.max_query_len) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
  if (tok0 >= q_len) return;  // nothing of this request here (uniform: the whole CTA leaves)

  const TileSpan spanA = tile_span(tok0, TOK, q_len, seq_len, p.causal);
  const TileSpan spanB = tile_span(tok0 + TOK, TOK, q_len, seq_len, p.causal);
  // Iteration i covers key tile j0 + i. Under a sliding window, j0 is the tile holding the
  // oldest key the CTA's first query sees; tiles before it are never loaded.
  // In prefix mode the CTA covers key tiles [j0, j0 + prefix_tiles_per_split) of the prefix.
  const int j0 = kPrefix          ? r * p.prefix_tiles_per_split
                 : p.window > 0 ? max(0, spanA.first - p.window + 1) / kBN
                                : 0;
  const int endA = kPrefix ? min(spanA.n_kv, j0 + p.prefix_tiles_per_split) : spanA.n_kv;
  const int endB = kPrefix ? min(spanB.n_kv, j0 + p.prefix_tiles_per_split) : spanB.n_kv;
  const int nA = max(0, endA - j0);
  const int nB = spanB.n_kv > 0 ? max(0, endB - j0) : 0;
  const int n_kv = max(nA, nB);
  // A lone tile (the pair's second tile is empty: decodes, verify blocks, a prompt's last tokens):
  // tile B's score block doubles tile A's, so S(j + 1) runs on the tensor core during the softmax of
  // tile j, and Q_B's buffer with the spare shared memory holds a third K/V stage.
  constexpr bool kLoneOk = !kPrefix && kQ == 0;
  const bool lone = kLoneOk && nB == 0;
  const int n_stages = lone ? kLoneStages : kStages;
  using L = Layout<kD, kQ>;
  const int bs = p.block_size;
  const int pages_per_tile = kBN / bs;
  const int seq_pages = (seq_len + bs - 1) / bs;
  if (kPrefix && n_kv <= 0) {
    // no prefix keys in this range (a short or empty prefix): the neutral partial (0, -inf, 0)
    const int rows = min(2 * TOK, q_len - tok0) * G;
    for (int i = tid; i < rows * (kD / 4); i += blockDim.x) {
      const int row = i / (kD / 4), c = i % (kD / 4);
      const size_t slot = ((size_t)(q_start + tok0 + row / G) * p.slot_count + r) * p.num_q_heads + kvh * G + row % G;
      *reinterpret_cast<float4*>(p.ws_acc + slot * kD + c * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c == 0) {
        p.ws_ml[slot * 2] = -INFINITY;
        p.ws_ml[slot * 2 + 1] = 0.f;
      }
    }
    return;
  }

  const int warp = tid >> 5, lane = tid & 31;
  // a kernel launched to overlap this one (it reads nothing this one writes) may start now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < kLoneStages; ++s) {
      // 8-bit caches: the producer's 32 lanes' scale copies arrive on the full barriers too
      mbar_init(&bars[B_KF + s], kQ != 0 ? 33 : 1);
      mbar_init(&bars[B_VF + s], kQ != 0 ? 33 : 1);
      mbar_init(&bars[B_KE + s], 1);
      mbar_init(&bars[B_VE + s], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_KR + s], 64);
      mbar_init(&bars[B_VR + s], 64);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[B_SF + t], 1);
      mbar_init(&bars[B_PR + t], kBM);
      mbar_init(&bars[B_OD + t], 1);
    }
    mbar_init(&bars[B_FIN], 1);
    fence_barrier_init();
    *abort_flag = 0;
    *issued_k = 0;
    *issued_v = 0;
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------ producer (warp 8): Q_A, Q_B once, then K/V
    // tiles. Lane k copies page k of a tile (its id loaded one tile ahead), so a tile's copies
    // go out from up to 8 threads at once: one thread issuing them all is slower than HBM at
    // small block sizes.
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(&bars[B_Q], (lone ? 1 : 2) * kTileBytes);
      for (int t = 0; t < (lone ? 1 : 2); ++t)
        for (int a = 0; a < kBlocks; ++a)
          tma_load_3d(smem + kOffQ + t * kTileBytes + a * kRegion, &qmap, &bars[B_Q], a * 64, kvh * G,
                      q_start + tok0 + t * TOK);
    }
    const int32_t* table = p.block_tables + (size_t)(kPrefix ? 0 : r) * p.max_blocks;
    // this lane's page of tile i (pages_per_tile <= 8 since the block size is >= 16)
    auto page_of = [&](int i) {
      const int pg = (j0 + i) * pages_per_tile + lane;
      return (lane < pages_per_tile && pg < seq_pages) ? __ldg(table + pg) : 0;
    };
    // 8-bit caches: a tile's 128 key (or value) scales, 4 per lane, copied asynchronously into
    // shared memory with completion on the tile's full barrier; positions past the sequence end,
    // or on a page outside the pool, are zero-filled instead of read
    auto copy_scales = [&](int i, int st, int page, const float* base, float* dst, uint64_t* bar) {
      const int key = 4 * lane;
      const int pg = __shfl_sync(0xffffffffu, page, key / bs);  // the lane holding this key's page
      const int pos0 = (j0 + i) * kBN + key;
      const bool pg_ok = pg >= 0 && pg < p.num_blocks;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool take = pg_ok && pos0 + e < seq_len;
        const float* src = take ? base + ((size_t)pg * bs + (key + e) % bs) * p.num_kv_heads + kvh : base;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst + st * 256 + key + e)),
                     "l"(src), "r"(take ? 4 : 0)
                     : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
    };
    float* scales = reinterpret_cast<float*>(smem + kOffScale);  // [stage][K 128 | V 128]
    // Copies of tile i go to stage i % n_stages once the tensor core has released the stage's
    // previous tile. A lone tile's K copies run one tile ahead of its V copies: a V stage frees
    // only after its P.V, and K(i + 1) would otherwise wait behind V(i) for it.
    const int lead = lone ? 1 : 0;
    auto copy_tile = [&](bool is_v, int i, int page) -> bool {
      const int st = i % n_stages;
      const int p0 = (j0 + i) * pages_per_tile;
      const int np = min(p0 + pages_per_tile, seq_pages) - p0;
      const uint32_t bytes = (uint32_t)np * bs * (uint32_t)(kQ != 0 ? kD : kD * 2);
      uint64_t* full = &bars[(is_v ? B_VF : B_KF) + st];
      if (i >= n_stages && !warp_wait(&bars[(is_v ? B_VE : B_KE) + st], ((i / n_stages) - 1) & 1, abort_flag))
        return false;
      if (lane == 0) mbar_arrive_expect_tx(full, bytes);
      __syncwarp();
      uint8_t* dst = smem + (is_v ? L::v_stage(st) : L::k_stage(st));
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      if (lane < np) {
        if (!is_v && (page < 0 || page >= p.num_blocks)) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // reads zeros
        if constexpr (kQ != 0) {  // the page's codes: one 128-byte row per key, into column block 1
          tma_load_4d(dst + kRegion + lane * bs * 128, map, full, 0, kvh, 0, page);
        } else if constexpr (L::kWide) {  // the whole page (bs / 8 row groups) in one copy
          tma_load_5d(dst + L::at(lane * bs, 0), map, full, 0, 0, 0, page * (bs / 8), kvh);
        } else {
          for (int a = 0; a < kBlocks; ++a) tma_load_4d(dst + a * kRegion + lane * bs * 128, map, full, a * 64, kvh, 0, page);
        }
      }
      if constexpr (kQ != 0) copy_scales(i, st, page, is_v ? p.v_scales : p.k_scales, is_v ? scales + 128 : scales, full);
      __syncwarp();
      if (lane == 0) *(is_v ? issued_v : issued_k) = i + 1;
      return true;
    };
    int cur = n_kv > 0 ? page_of(0) : 0, prev = 0;  // this lane's page of tile e, of tile e - 1
    for (int e = 0; e < n_kv + lead; ++e) {
      const int nxt = e + 1 < n_kv ? page_of(e + 1) : 0;
      if (e < n_kv && !copy_tile(false, e, cur)) {
        if (lane == 0) set_abort(abort_flag, p.err);
        break;
      }
      if (e - lead >= 0 && !copy_tile(true, e - lead, lead ? prev : cur)) {
        if (lane == 0) set_abort(abort_flag, p.err);
        break;
      }
      prev = cur;
      cur = nxt;
    }
  } else if (warp == 9) {
    // ------------------------------------------------ MMA issuer (lane 0); the warp zeroes V tails
    const uint32_t id_s = idesc_bf16(kBM, kBN, false);
    const uint32_t id_pv = idesc_bf16(kBM, kD, true);
    const uint32_t sQ = smem_addr(smem + kOffQ);
    const uint32_t sK = smem_addr(smem + kOffK);
    const uint32_t sV = smem_addr(smem + kOffV);
    // Descriptors advance by adding (byte offset >> 4) to the start-address field; every
    // operand lies below 256 KiB of the shared window, so the 14-bit field never carries.
    const uint64_t dq0 = sdesc(sQ, 16, 1024);
    const uint64_t dk0 = sdesc(sK, 16, L::kSBO);
    const uint64_t dv0 = sdesc(sV, L::kCB, L::kSBO);  // MN-major V: 64-column blocks L::kCB apart
    if (lone) {
      // a lone tile: the two softmax groups take the key tiles in turn (tile j: group j & 1, its
      // score block and its O block), so two softmaxes run at once. Issue order S(0), S(1), then
      // per tile P.V(j), S(j + 2).
      auto dk_of = [&](int st) { return sdesc(smem_addr(smem + L::k_stage(st)), 16, L::kSBO); };
      auto dv_of = [&](int st) { return sdesc(smem_addr(smem + L::v_stage(st)), L::kCB, L::kSBO); };
      // S(j) into block j & 1, then release its K stage (only if the producer will refill it)
      auto issue_s1 = [&](int j) {
        if (lane == 0) {
          const uint64_t dk = dk_of(j % kLoneStages);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t offq = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
            const uint64_t offk = (uint64_t)(((kk >> 2) * L::kCB + (kk & 3) * 32) >> 4);
            umma_ss(tmem + col_s(j & 1), dq0 + offq, dk + offk, id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars[B_SF + (j & 1)]);
          if (j + kLoneStages < nA) umma_commit(&bars[B_KE + j % kLoneStages]);
        }
      };
      bool ok = warp_wait(&bars[B_Q], 0, abort_flag);
      for (int j = 0; ok && j < min(2, nA); ++j) {
        if (!(ok = warp_wait(&bars[B_KF + j], 0, abort_flag))) break;
        tc_fence_after();
        issue_s1(j);
        __syncwarp();
      }
      for (int j = 0; ok && j < nA; ++j) {
        const int st = j % kLoneStages;
        if (!(ok = warp_wait(&bars[B_VF + st], (j / kLoneStages) & 1, abort_flag))) break;
        const int zero_from = seq_len - (j0 + j) * kBN;  // V rows at or past the sequence end: exact zeros
        if (zero_from < kBN) {
          uint8_t* vbp = smem + L::v_stage(st);
          const int rows = kBN - zero_from;
          for (int i = lane; i < rows * (kD / 8); i += 32) {
            const int row = zero_from + i / (kD / 8), c = i % (kD / 8);
            *reinterpret_cast<uint4*>(vbp + L::at(row, c >> 3) + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
        }
        if (!(ok = warp_wait(&bars[B_PR + (j & 1)], (j >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv = dv_of(st);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(tmem + col_o<kD>(j & 1), tmem + col_s(j & 1) + 8 * kk, dv + (uint64_t)((kk * 2 * L::kSBO) >> 4),
                    id_pv, (j > 1 || kk > 0) ? 1u : 0u);
          umma_commit(&bars[B_OD + (j & 1)]);
          if (j + kLoneStages < nA) umma_commit(&bars[B_VE + st]);
        }
        // S(j + 2) overwrites P(j) in block j & 1: it is issued after P.V(j), which reads it first
        if (j + 2 < nA) {
          if (!(ok = warp_wait(&bars[B_KF + (j + 2) % kLoneStages], ((j + 2) / kLoneStages) & 1, abort_flag))) break;
          tc_fence_after();
          issue_s1(j + 2);
        }
        __syncwarp();
      }
      if (!ok) set_abort(abort_flag, p.err);
    } else {
      // S_t(j) = Q_t K_j^T into S block t
      auto issue_s = [&](int t, int j) {
        if (lane == 0) {
          const uint64_t dq = dq0 + (uint64_t)((t * kTileBytes) >> 4);
          const uint64_t dk = dk0 + (uint64_t)(((j % kStages) * kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t offq = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
            const uint64_t offk = (uint64_t)(((kk >> 2) * L::kCB + (kk & 3) * 32) >> 4);
            umma_ss(tmem + col_s(t), dq + offq, dk + offk, id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars[B_SF + t]);
        }
      };
      // O_t += P_t(j) V_j (N = kD: every 64-column block of V), P_t from the first 64 TMEM
      // columns of S block t
      auto issue_pv = [&](int t, int j) {
        if (lane == 0) {
          const uint64_t dv = dv0 + (uint64_t)(((j % kStages) * kTileBytes) >> 4);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(tmem + col_o<kD>(t), tmem + col_s(t) + 8 * kk, dv + (uint64_t)((kk * 2 * L::kSBO) >> 4), id_pv,
                    kk > 0 ? 1u : acc0);
          umma_commit(&bars[B_OD + t]);
        }
      };
      auto commit_if = [&](bool cond, int bar) {
        if (cond && lane == 0) umma_commit(&bars[bar]);
      };
      // 8-bit caches: a tile is ready for the tensor core once the converters have dequantised it
      constexpr int kReadyK = kQ != 0 ? B_KR : B_KF;
      constexpr int kReadyV = kQ != 0 ? B_VR : B_VF;
      bool ok = warp_wait(&bars[B_Q], 0, abort_flag) && warp_wait(&bars[kReadyK], 0, abort_flag);
      if (ok) {
        tc_fence_after();
        if (nA > 0) issue_s(0, 0);
        if (nB > 0) issue_s(1, 0);
        commit_if(kStages < n_kv, B_KE + 0);
        __syncwarp();
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % kStages;
        if (!(ok = warp_wait(&bars[kReadyV + st], (j / kStages) & 1, abort_flag))) break;
        const int zero_from = seq_len - (j0 + j) * kBN;  // V rows at or past the sequence end: exact zeros
        if (kQ == 0 && zero_from < kBN) {  // (8-bit caches: the converters write those rows as zeros)
          uint8_t* vbp = smem + kOffV + st * kTileBytes;
          const int rows = kBN - zero_from;
          for (int i = lane; i < rows * (kD / 8); i += 32) {
            const int row = zero_from + i / (kD / 8), c = i % (kD / 8);
            *reinterpret_cast<uint4*>(vbp + L::at(row, c >> 3) + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
        }
        if (j < nA) {
          if (!(ok = warp_wait(&bars[B_PR + 0], j & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(0, j);
        }
        const bool next = j + 1 < n_kv;
        if (next) {
          if (!(ok = warp_wait(&bars[kReadyK + (j + 1) % kStages], ((j + 1) / kStages) & 1, abort_flag))) break;
          tc_fence_after();
          if (j + 1 < nA) issue_s(0, j + 1);
        }
        if (j < nB) {
          if (!(ok = warp_wait(&bars[B_PR + 1], j & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(1, j);
        }
        // release V_j, then issue S_B(j+1) and release K_{j+1}, each only if the producer will
        // refill that stage (an arrive nobody waits for could land after this CTA has left)
        commit_if(j + kStages < n_kv, B_VE + st);
        if (next) {
          if (j + 1 < nB) issue_s(1, j + 1);
          commit_if(j + 1 + kStages < n_kv, B_KE + (j + 1) % kStages);
        }
        __syncwarp();
      }
      if (!ok) set_abort(abort_flag, p.err);
    }
  } else if (kQ != 0 && warp >= 10) {
    // ------------------------------------------------ 8-bit caches: warps 10-11 dequantise each
    // K and V tile in place ("32. Production attention kernels", Quantized KV caches: the tile of
    // codes times its per-slot scale, then used exactly like a bf16 tile): thread c takes rows c
    // and c + 64; rows at or past the sequence end become zeros (a stale slot may hold anything)
    const int c = tid - 320;
    const float* scales = reinterpret_cast<const float*>(smem + kOffScale);
    bool ok = true;
    for (int i = 0; ok && i < n_kv; ++i) {
      const int st = i % kStages;
      const int key0 = (j0 + i) * kBN;
      for (int kv = 0; kv < 2; ++kv) {
        if (!warp_wait(&bars[(kv ? B_VF : B_KF) + st], (i / kStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* tile = smem + (kv ? kOffV : kOffK) + st * kTileBytes;
        const float* sc = scales + st * 256 + kv * 128;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int row = c + 64 * h;
          const bool valid = key0 + row < seq_len;
          dequantize_row<kQ>(tile, row, valid ? sc[row] : 0.f, valid);
        }
        fence_async_smem();  // generic-proxy writes, read next by the tensor core
        mbar_arrive(&bars[(kv ? B_VR : B_KR) + st]);
      }
    }
    if (!ok) set_abort(abort_flag, p.err);
  } else {
    // ------------------------------------------------ softmax: warps 0-3 tile A, 4-7 tile B
    // (a lone tile: both groups on tile A's rows, group t taking key tiles t, t + 2, ... into
    // O block t; group 0 merges the two at the end)
    const int t = warp >> 2;
    const int n_mine = lone ? (nA + 1 - t) / 2 : (t == 0 ? nA : nB);
    const int row = tid & (kBM - 1);
    const int tok = tok0 + (lone ? 0 : t) * TOK + row / G;
    const bool row_valid = tok < q_len;
    const int qpos = seq_len - q_len + tok;
    const int vis_end = p.causal ? min(qpos + 1, seq_len) : seq_len;
    const int vis_start = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
    const bool capped = p.softcap_log2 > 0.f;
    const float c = p.scale_log2;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + col_s(t);
    const uint32_t o_col = lane_base + col_o<kD>(t);
    // a sink logit starts the running state: it joins the denominator and adds no value (a lone
    // tile: in group 0's state only)
    const bool sink = p.sinks != nullptr && !(lone && t == 1);
    float m_run = sink ? p.sinks[kvh * G + row % G] * kLog2e : -INFINITY;
    float l_run = sink ? 1.f : 0.f;
    bool ok = true;
    for (int k = 0; k < n_mine; ++k) {
      const int j = lone ? 2 * k + t : k;  // the key tile (counted from j0)
      if (!warp_wait(&bars[B_SF + t], k & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nvis = vis_end - (j0 + j) * kBN;  // keys below this index of the tile are not too new
      const int nlo = vis_start - (j0 + j) * kBN;  // keys from this index on are inside the window
      const bool full = nvis >= kBN && nlo <= 0;
      // the row's 128 scores, one TMEM round trip (tcgen05.wait::ld waits for every load)
      uint32_t sv[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(s_col + 32 * q4, sv[q4]);
      tmem_ld_wait();
      if (!full) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; ++i)  // select: NaN past the sequence end never survives
            sv[q4][i] = (q4 * 32 + i < nvis && q4 * 32 + i >= nlo) ? sv[q4][i] : __float_as_uint(-INFINITY);
      }
      // row maximum over eight interleaved chains (short dependency chains)
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sv[q4][i]));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // the softcap is increasing, so the capped maximum is the cap of the maximum
      const float mxs = capped ? (mx == -INFINITY ? -INFINITY : p.softcap_log2 * tanh_ex2(mx * p.scale_over_cap))
                               : mx * c;
      float m_new = m_run, alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY || mxs > m_run + kRescaleThreshold) {
        m_new = mxs;
        alpha = exp2f(m_run - (m_new == -INFINITY ? 0.f : m_new));
        rescale = (k > 0);
      }
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      // probabilities, packed to bf16 pairs over the score columns already consumed
      // (keys 64h..64h+63 -> columns 32h..32h+31)
      const uint64_t c2 = f2(c, c), nmu2 = f2(-mu, -mu);
      uint64_t sum2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t* src = sv[2 * h + (i >> 4)];
          const int e = (2 * i) & 31;
          float x0, x1;
          if (capped) {  // masked keys hold -inf: tanh gives -1, the select below zeroes them
            x0 = p.softcap_log2 * tanh_ex2(__uint_as_float(src[e]) * p.scale_over_cap) - mu;
            x1 = p.softcap_log2 * tanh_ex2(__uint_as_float(src[e + 1]) * p.scale_over_cap) - mu;
            x0 = __uint_as_float(src[e]) == -INFINITY ? -INFINITY : x0;
            x1 = __uint_as_float(src[e + 1]) == -INFINITY ? -INFINITY : x1;
          } else {
            f2_split(f2_fma(f2(__uint_as_float(src[e]), __uint_as_float(src[e + 1])), c2, nmu2), x0, x1);
          }
          const float p0 = ex2(x0), p1 = ex2(x1);  // 2^-inf = 0 for masked keys
          sum2[i & 1] = f2_add(sum2[i & 1], f2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);  // key 64h + 2i in the low half, 64h + 2i + 1 in the high half
        }
        tmem_st32(s_col + 32 * h, pk);
      }
      float la, lb;
      f2_split(f2_add(sum2[0], sum2[1]), la, lb);
      const float lsum = la + lb;
      l_run = l_run * alpha + lsum;
      m_run = m_new;
      // this S has landed, so the P.V into O_t before it (issued earlier) is complete: O is stable
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll
        for (int q4 = 0; q4 < kD / 32; ++q4) {
          uint32_t ov[32];
          tmem_ld32(o_col + 32 * q4, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
          tmem_st32(o_col + 32 * q4, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_PR + t]);
    }
    // the last P.V of this tile
    if (ok && n_mine > 0 && !warp_wait(&bars[B_OD + t], (n_mine - 1) & 1, abort_flag)) ok = false;
    // a lone tile of two or more key tiles: group 1 hands its rows' (m, l) to group 0, which merges
    // O block 1 into its own. Group 1's last P.V was issued after every S, so K stage 0 is free.
    const bool merge = lone && nA > 1;
    float m_o = -INFINITY, l_o = 0.f;
    if (merge) {
      float* xch = reinterpret_cast<float*>(smem + L::k_stage(0));
      if (t == 1) {
        xch[row] = m_run;
        xch[kBM + row] = l_run;
        asm volatile("bar.arrive 2, 256;" ::: "memory");
      } else {
        asm volatile("bar.sync 2, 256;" ::: "memory");
        m_o = xch[row];
        l_o = xch[kBM + row];
      }
    }
    if (!ok) {
      set_abort(abort_flag, p.err);
    } else if (kPrefix) {
      // cascade prefix pass: the row's unnormalised partial (acc, m in log2 units, l) in the
      // split-partial layout the combine merges. (A tile without keys here has no valid rows:
      // ranges past the prefix end left the kernel at the top.)
      // The accumulator rows go out through this tile's Q buffer (every S of the tile has read
      // it): each warp stages 32 columns of its 32 rows, then writes them 4 rows of 128 bytes per
      // instruction instead of one 16-byte piece of each of 32 rows.
      const size_t slot = ((size_t)(q_start + tok) * p.slot_count + r) * p.num_q_heads + kvh * G + row % G;
      if (n_mine > 0) {
        tc_fence_after();
        uint8_t* stage = smem + kOffQ + t * kTileBytes + (warp & 3) * (32 * 128);
        const int piece = lane & 7;
#pragma unroll 1
        for (int q4 = 0; q4 < kD / 32; ++q4) {
          uint32_t ov[32];
          tmem_ld32(o_col + 32 * q4, ov);
          tmem_ld_wait();
#pragma unroll
          for (int pc = 0; pc < 8; ++pc)  // 128-byte rows, 16-byte pieces swizzled by the row
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((pc ^ (lane & 7)) << 4)) =
                make_uint4(ov[4 * pc], ov[4 * pc + 1], ov[4 * pc + 2], ov[4 * pc + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3);     // the warp's row this lane copies a piece of
            const int trow = (warp & 3) * 32 + rr;  // its row in the tile
            const int rtok = tok0 + t * TOK + trow / G;
            if (rtok < q_len) {
              const size_t rslot =
                  ((size_t)(q_start + rtok) * p.slot_count + r) * p.num_q_heads + kvh * G + trow % G;
              *reinterpret_cast<uint4*>(p.ws_acc + rslot * kD + q4 * 32 + piece * 4) =
                  *reinterpret_cast<const uint4*>(stage + rr * 128 + ((piece ^ (rr & 7)) << 4));
            }
          }
          __syncwarp();
        }
        if (row_valid) {
          p.ws_ml[slot * 2] = m_run;
          p.ws_ml[slot * 2 + 1] = l_run;
        }
      }
    } else if (n_mine > 0 && !(lone && t == 1)) {
      tc_fence_after();
      // O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)), m the larger
      float a0 = 1.f, a1 = 0.f, l = l_run;
      if (merge) {
        const float m = fmaxf(m_run, m_o);
        const float mu = m == -INFINITY ? 0.f : m;
        a0 = exp2f(m_run - mu);
        a1 = exp2f(m_o - mu);
        l = l_run * a0 + l_o * a1;
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float s0 = a0 * inv, s1 = a1 * inv;
      const uint32_t o1_col = lane_base + col_o<kD>(1);
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(q_start + tok) * p.out_stride +
                           (size_t)(kvh * G + row % G) * kD;
#pragma unroll
      for (int q4 = 0; q4 < kD / 32; ++q4) {
        uint32_t ov[32];
        float o[32];
        tmem_ld32(o_col + 32 * q4, ov);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(ov[i]) * s0;
        if (merge) {
          tmem_ld32(o1_col + 32 * q4, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = fmaf(__uint_as_float(ov[i]), s1, o[i]);
        }
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(o[i], o[i + 1]);
            w.y = pack_bf16x2(o[i + 2], o[i + 3]);
            w.z = pack_bf16x2(o[i + 4], o[i + 5]);
            w.w = pack_bf16x2(o[i + 6], o[i + 7]);
            *reinterpret_cast<uint4*>(out + q4 * 32 + i) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // drain: every MMA this CTA issued, every copy still landing
    if (warp == 9 && lane == 0) {
      umma_commit(&bars[B_FIN]);
      (void)mbar_wait(&bars[B_FIN], 0);
    }
    if (warp == 8 && lane == 0) {
      (void)mbar_wait(&bars[B_Q], 0);
      const int ik = *issued_k, iv = *issued_v;
      for (int j = max(0, ik - n_stages); j < ik; ++j) (void)mbar_wait(&bars[B_KF + j % n_stages], (j / n_stages) & 1);
      for (int j = max(0, iv - n_stages); j < iv; ++j) (void)mbar_wait(&bars[B_VF + j % n_stages], (j / n_stages) & 1);
    }
    __syncthreads();
  }
  if (warp == 9) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

bool varlen_tc_supported(int head_dim, int group, int block_size) {
  const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8 || group == 16;
  const bool bs_ok = block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128;
  return (head_dim == 64 || head_dim == 128 || head_dim == 256) && g_ok && bs_ok;
}

bool varlen_tc_prefix_supported(int head_dim, int group, int block_size) {
  return head_dim != 256 && varlen_tc_supported(head_dim, group, block_size);
}

int varlen_tc_tokens_per_cta(int group) { return 2 * (kBM / group); }

namespace {

// ---------------------------------------------------------------- device-side work list
// The planned grid's work list, built on the GPU from the batch's lengths as they are when the
// call runs (so a captured graph follows them): every (tile pair, request) item the batch has,
// longest first by its key-tile count ("TileInfer.jl - Attention kernels", Open questions:
// heaviest causal blocks first), then -1 up to the grid's capacity. One CTA: a histogram of the
// items' key-tile counts, a descending scan, and a scatter (the order among items of equal
// count is not fixed; each item computes the same result wherever it runs).
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 4096;  // counts of 4095 key tiles and more share the last bucket

struct PlanArgs {
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  int32_t* items;
  int32_t* err;
  int num_reqs;
  int num_tokens;
  int tok_tile;  // tokens of one 128-row query tile (128 / group)
  int q_tiles;   // tile pairs per request in the grid's index space
  int causal;
  int window;
  int skip_upto;
  int capacity;
};

// Key tiles of pair t of request r (its larger tile's count), or -1 if the pair is no item: the
// request is empty, served by the split-KV decode, or has fewer queries.
__device__ int plan_pair_work(const PlanArgs& a, int r, int t) {
  const int start = a.query_start_loc[r], stop = a.query_start_loc[r + 1];
  const int q_len = stop - start;
  if (q_len <= 0) return -1;
  if (start >= 0 && stop <= a.num_tokens && q_len <= a.skip_upto) return -1;
  const int tok0 = t * 2 * a.tok_tile;
  if (tok0 >= q_len) return -1;
  const int seq = a.seq_lens[r];
  int w = 0;
  for (int h = 0; h < 2; ++h) {
    const int t0 = tok0 + h * a.tok_tile;
    const int n = max(0, min(a.tok_tile, q_len - t0));
    if (n == 0) continue;
    const int first = seq - q_len + t0;
    const int key_end = a.causal ? min(seq, first + n) : seq;
    const int j0 = a.window > 0 ? max(0, first - a.window + 1) / 128 : 0;
    w = max(w, (max(0, key_end) + 127) / 128 - j0);
  }
  return max(0, w);
}

__global__ void __launch_bounds__(kPlanThreads) varlen_plan_kernel(const __grid_constant__ PlanArgs a) {
  __shared__ int start[kPlanBuckets];
  __shared__ int warp_sums[kPlanThreads / 32];
  __shared__ int total;
  // the tensor-core grid launched after this kernel may start now; it waits for this grid's
  // completion before it reads the list
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x;
  for (int b = tid; b < kPlanBuckets; b += kPlanThreads) start[b] = 0;
  __syncthreads();
  const long long pairs = (long long)a.num_reqs * a.q_tiles;
  for (long long i = tid; i < pairs; i += kPlanThreads) {
    const int r = (int)(i / a.q_tiles), t = (int)(i % a.q_tiles);
    const int w = plan_pair_work(a, r, t);
    if (w >= 0) atomicAdd(&start[min(w, kPlanBuckets - 1)], 1);
  }
  __syncthreads();
  // exclusive scan over the buckets in descending order: thread k owns buckets
  // kPlanBuckets - 1 - 4k - c (c = 0..3); start[b] becomes the first slot of bucket b
  constexpr int kPer = kPlanBuckets / kPlanThreads;
  int cnt[kPer], run = 0;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    cnt[c] = start[kPlanBuckets - 1 - (tid * kPer + c)];
    run += cnt[c];
  }
  const int lane = tid & 31, warp = tid >> 5;
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int ws = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, ws, o);
      if (lane >= o) ws += v;
    }
    warp_sums[lane] = ws;  // inclusive over warps
    if (lane == 31) total = ws;
  }
  __syncthreads();
  int off = incl - run + (warp > 0 ? warp_sums[warp - 1] : 0);
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    start[kPlanBuckets - 1 - (tid * kPer + c)] = off;
    off += cnt[c];
  }
  __syncthreads();
  for (long long i = tid; i < pairs; i += kPlanThreads) {
    const int r = (int)(i / a.q_tiles), t = (int)(i % a.q_tiles);
    const int w = plan_pair_work(a, r, t);
    if (w < 0) continue;
    const int pos = atomicAdd(&start[min(w, kPlanBuckets - 1)], 1);
    if (pos < a.capacity)
      a.items[pos] = t * a.num_reqs + r;
    else
      flag_error(a.err, PA_ERRBIT_QUERY_LAYOUT);  // more items than the grid's bound: a malformed layout
  }
  for (int i = total + tid; i < a.capacity; i += kPlanThreads) a.items[i] = -1;
}

template <bool kPrefix, int kD, int kQ = 0>
cudaError_t launch_pair(const VarlenParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                        const CUtensorMap& vmap, long long ctas, cudaStream_t stream) {
  // the shared-memory opt-in is per device and kernel; setting it twice is harmless
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  constexpr int smem = Layout<kD, kQ>::kSmemBytes;
  constexpr int threads = kQ != 0 ? kThreadsQ : kThreads;
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(varlen_tc_kernel<kPrefix, kD, kQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  if (!p.plan_on_device) {
    varlen_tc_kernel<kPrefix, kD, kQ><<<(unsigned)ctas, threads, smem, stream>>>(p, qmap, kmap, vmap);
    return cudaGetLastError();
  }
  return launch_dependent(varlen_tc_kernel<kPrefix, kD, kQ>, (unsigned)ctas, threads, smem, stream, p, qmap, kmap,
                          vmap);
}
}  // namespace

long long varlen_device_plan_capacity(int num_reqs, int num_tokens, int max_query_len, int group, int skip_upto) {
  const int per_cta = varlen_tc_tokens_per_cta(group);
  const long long q_tiles = (max_query_len + per_cta - 1) / per_cta;
  // a request with q queries has cdiv(q, per_cta) <= q / per_cta + 1 pairs; the queries of the
  // requests add up to num_tokens, and with short requests skipped a planned request has more
  // than skip_upto queries
  const long long planned_reqs =
      std::min<long long>(num_reqs, skip_upto > 0 ? num_tokens / (skip_upto + 1) : num_reqs);
  return std::min<long long>((long long)num_reqs * q_tiles, num_tokens / per_cta + planned_reqs);
}

cudaError_t launch_varlen_device_plan(const int32_t* query_start_loc, const int32_t* seq_lens, int num_reqs,
                                      int num_tokens, int group, int q_tiles, int causal, int window, int skip_upto,
                                      int32_t* items, int capacity, int32_t* err, cudaStream_t stream) {
  PlanArgs a;
  a.query_start_loc = query_start_loc;
  a.seq_lens = seq_lens;
  a.items = items;
  a.err = err;
  a.num_reqs = num_reqs;
  a.num_tokens = num_tokens;
  a.tok_tile = kBM / group;
  a.q_tiles = q_tiles;
  a.causal = causal;
  a.window = window;
  a.skip_upto = skip_upto;
  a.capacity = capacity;
  varlen_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_varlen_tc(const VarlenParams& p_in, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  VarlenParams p = p_in;
  if (p.out_stride == 0) p.out_stride = (long long)p.num_q_heads * p.head_dim;  // dense rows
  const long long ctas = (p.work_items != nullptr && !p.prefix_mode ? (long long)p.num_items
                                                                     : (long long)p.q_tiles * p.num_reqs) *
                         p.num_kv_heads;
  if (ctas <= 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (p.quant != 0) {  // 8-bit caches: head_dim 128, the two-tile kernel with its converter warps
    if (p.head_dim != 128 || p.prefix_mode) return cudaErrorInvalidValue;
    return p.quant == 1 ? launch_pair<false, 128, 1>(p, qmap, kmap, vmap, ctas, stream)
                        : launch_pair<false, 128, 2>(p, qmap, kmap, vmap, ctas, stream);
  }
  if (p.head_dim == 256) {
    if (p.prefix_mode) return cudaErrorInvalidValue;
    return launch_varlen_tc256(p, qmap, kmap, vmap, ctas, stream);
  }
  if (p.head_dim == 64)
    return p.prefix_mode ? launch_pair<true, 64>(p, qmap, kmap, vmap, ctas, stream)
                         : launch_pair<false, 64>(p, qmap, kmap, vmap, ctas, stream);
  if (p.head_dim == 128)
    return p.prefix_mode ? launch_pair<true, 128>(p, qmap, kmap, vmap, ctas, stream)
                         : launch_pair<false, 128>(p, qmap, kmap, vmap, ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
