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
#include <atomic>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kBM = 128;  // packed query rows per tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kD = 128;   // head dim of this kernel
constexpr int kStages = 2;
constexpr int kRegion = 128 * 128;       // one [128 rows][64 bf16] swizzled column half: 16 KiB
constexpr int kTileBytes = 2 * kRegion;  // a 128 x 128 bf16 tile
constexpr int kOffQ = 0;                 // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffBar = kOffV + kStages * kTileBytes;
enum {
  B_Q = 0,
  B_KF = 1,   // +stage
  B_VF = 3,   // +stage
  B_KE = 5,   // +stage
  B_VE = 7,   // +stage
  B_SF = 9,   // +tile (A, B)
  B_PR = 11,  // +tile
  B_OD = 13,  // +tile
  B_FIN = 15,
  kNumBars = 16
};
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 32;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
// TMEM columns of tile t's score block and output accumulator
__host__ __device__ constexpr uint32_t col_s(int t) { return t == 0 ? 0u : 128u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t == 0 ? 256u : 384u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// ---------------------------------------------------------------- tcgen05 helpers
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major, B K-major
// or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets (>> 4), the
// sm_100 descriptor version (1 at bit 46) and the 128-byte swizzle mode (2 at bit 61).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem); A is M rows on the TMEM lanes, two bf16 per column.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#define PA_R32(v) \
  "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), \
  "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),       \
  "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),      \
  "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
#define PA_W32(v) \
  "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), \
  "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),   \
  "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),   \
  "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])

// 32 consecutive columns of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PA_R32(v)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      PA_W32(v)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Bounded wait that also gives up as soon as another role has aborted. The clock and the
// abort flag are checked once per 64 polls so that waiting warps take few issue slots.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- softmax arithmetic
// 2^x on the special-function unit (flushes results below 2^-126 to zero: such
// probabilities are far below bf16 resolution against the row maximum's 1).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs (Blackwell f32x2 arithmetic: one instruction for two lanes of work).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// tanh(y) = 1 - 2 / (2^(2 y log2 e) + 1): one ex2 and one approximate reciprocal; absolute
// error ~1e-7 (the softcap multiplies it by the cap), exact limits +-1 at +-infinity.
__device__ __forceinline__ float tanh_ex2(float y) {
  const float e = ex2(y * 2.8853900817779268f);
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
  return 1.f - 2.f * r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The same, with one verdict for the whole warp, so that a warp either proceeds to its
// warp-collective tcgen05 instructions together or leaves together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = wait_or_abort(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag, int32_t* err) {
  *abort_flag = 1;
  flag_error(err, PA_ERRBIT_WAIT_TIMEOUT);
}

struct TileSpan {
  int n_tok;    // valid query tokens in the tile (0 = tile unused)
  int first;    // position of the tile's first query
  int n_kv;     // 128-key tiles it needs
};

__device__ __forceinline__ TileSpan tile_span(int tok0, int TOK, int q_len, int seq_len, int causal) {
  TileSpan t;
  t.n_tok = max(0, min(TOK, q_len - tok0));
  t.first = seq_len - q_len + tok0;
  const int key_end = causal ? min(seq_len, t.first + t.n_tok) : seq_len;
  t.n_kv = t.n_tok > 0 ? (key_end + kBN - 1) / kBN : 0;
  return t;
}

// kPrefix: the cascade's shared-prefix pass (one request of num_tokens query rows that all
// see the whole prefix; unnormalised partials out instead of normalised rows).
template <bool kPrefix>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_tc_kernel(const __grid_constant__ VarlenParams p, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_tiles = reinterpret_cast<int*>(tmem_slot + 2);

  // ---- which tile pair: from the caller's plan (heaviest first by the host's estimate, no empty
  // pairs), else heaviest (last) query tiles first across all requests and heads
  int tile, r, kvh;  // r: the request, or the prefix key range in prefix mode
  if (!kPrefix && p.work_items != nullptr) {
    const int item = __ldg(p.work_items + blockIdx.x / p.num_kv_heads);
    kvh = (int)(blockIdx.x % p.num_kv_heads);
    tile = item / p.num_reqs;
    r = item - tile * p.num_reqs;
    if (item < 0 || tile >= p.q_tiles) {  // not an item of this batch: nothing to do here
      if (threadIdx.x == 0 && kvh == 0) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
      return;
    }
  } else {
    const int per_tile = p.num_reqs * p.num_kv_heads;
    tile = p.q_tiles - 1 - (int)(blockIdx.x / per_tile);
    const int rem = (int)(blockIdx.x % per_tile);
    r = rem / p.num_kv_heads;
    kvh = rem - r * p.num_kv_heads;
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_KF + s], 1);
      mbar_init(&bars[B_VF + s], 1);
      mbar_init(&bars[B_KE + s], 1);
      mbar_init(&bars[B_VE + s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[B_SF + t], 1);
      mbar_init(&bars[B_PR + t], kBM);
      mbar_init(&bars[B_OD + t], 1);
    }
    mbar_init(&bars[B_FIN], 1);
    fence_barrier_init();
    *abort_flag = 0;
    *issued_tiles = 0;
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
      mbar_arrive_expect_tx(&bars[B_Q], 2 * kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int a = 0; a < 2; ++a)
          tma_load_3d(smem + kOffQ + t * kTileBytes + a * kRegion, &qmap, &bars[B_Q], a * 64, kvh * G,
                      q_start + tok0 + t * TOK);
    }
    const int32_t* table = p.block_tables + (size_t)(kPrefix ? 0 : r) * p.max_blocks;
    // this lane's page of tile i (pages_per_tile <= 8 since the block size is >= 16)
    auto page_of = [&](int i) {
      const int pg = (j0 + i) * pages_per_tile + lane;
      return (lane < pages_per_tile && pg < seq_pages) ? __ldg(table + pg) : 0;
    };
    int cur = n_kv > 0 ? page_of(0) : 0;
    for (int i = 0; i < n_kv; ++i) {
      const int st = i % kStages;
      const uint32_t round_parity = ((i / kStages) - 1) & 1;
      const int p0 = (j0 + i) * pages_per_tile;
      const int np = min(p0 + pages_per_tile, seq_pages) - p0;
      const uint32_t bytes = (uint32_t)np * bs * 256u;
      const int nxt = i + 1 < n_kv ? page_of(i + 1) : 0;
      if (i >= kStages && !warp_wait(&bars[B_KE + st], round_parity, abort_flag)) {
        if (lane == 0) set_abort(abort_flag, p.err);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars[B_KF + st], bytes);
      __syncwarp();
      if (lane < np) {
        if (cur < 0 || cur >= p.num_blocks) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // reads zeros
        for (int a = 0; a < 2; ++a)
          tma_load_4d(smem + kOffK + st * kTileBytes + a * kRegion + lane * bs * 128, &kmap, &bars[B_KF + st],
                      a * 64, kvh, 0, cur);
      }
      if (i >= kStages && !warp_wait(&bars[B_VE + st], round_parity, abort_flag)) {
        if (lane == 0) {
          set_abort(abort_flag, p.err);
          *issued_tiles = i + 1;  // K of iteration i is in flight
        }
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars[B_VF + st], bytes);
      __syncwarp();
      if (lane < np)
        for (int a = 0; a < 2; ++a)
          tma_load_4d(smem + kOffV + st * kTileBytes + a * kRegion + lane * bs * 128, &vmap, &bars[B_VF + st],
                      a * 64, kvh, 0, cur);
      __syncwarp();
      if (lane == 0) *issued_tiles = i + 1;
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
    const uint64_t dk0 = sdesc(sK, 16, 1024);
    const uint64_t dv0 = sdesc(sV, kRegion, 1024);  // MN-major V: 64-column halves kRegion apart
    // S_t(j) = Q_t K_j^T into S block t
    auto issue_s = [&](int t, int j) {
      if (lane == 0) {
        const uint64_t dq = dq0 + (uint64_t)((t * kTileBytes) >> 4);
        const uint64_t dk = dk0 + (uint64_t)(((j % kStages) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
          umma_ss(tmem + col_s(t), dq + off, dk + off, id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_SF + t]);
      }
    };
    // O_t += P_t(j) V_j (N = 128: both 64-column halves of V), P_t from the first 64 TMEM
    // columns of S block t
    auto issue_pv = [&](int t, int j) {
      if (lane == 0) {
        const uint64_t dv = dv0 + (uint64_t)(((j % kStages) * kTileBytes) >> 4);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tmem + col_o(t), tmem + col_s(t) + 8 * kk, dv + (uint64_t)((kk * 2048) >> 4), id_pv,
                  kk > 0 ? 1u : acc0);
        umma_commit(&bars[B_OD + t]);
      }
    };
    auto commit_if = [&](bool cond, int bar) {
      if (cond && lane == 0) umma_commit(&bars[bar]);
    };
    bool ok = warp_wait(&bars[B_Q], 0, abort_flag) && warp_wait(&bars[B_KF], 0, abort_flag);
    if (ok) {
      tc_fence_after();
      if (nA > 0) issue_s(0, 0);
      if (nB > 0) issue_s(1, 0);
      commit_if(kStages < n_kv, B_KE + 0);
      __syncwarp();
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int st = j % kStages;
      if (!(ok = warp_wait(&bars[B_VF + st], (j / kStages) & 1, abort_flag))) break;
      const int zero_from = seq_len - (j0 + j) * kBN;  // V rows at or past the sequence end: exact zeros
      if (zero_from < kBN) {
        uint8_t* vbp = smem + kOffV + st * kTileBytes;
        const int rows = kBN - zero_from;
        for (int i = lane; i < rows * 16; i += 32) {
          const int row = zero_from + i / 16, c = i % 16;
          *reinterpret_cast<uint4*>(vbp + (c >> 3) * kRegion + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
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
        if (!(ok = warp_wait(&bars[B_KF + (j + 1) % kStages], ((j + 1) / kStages) & 1, abort_flag))) break;
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
  } else {
    // ------------------------------------------------ softmax: warps 0-3 tile A, 4-7 tile B
    const int t = warp >> 2;
    const int n_mine = t == 0 ? nA : nB;
    const int row = tid & (kBM - 1);
    const int tok = tok0 + t * TOK + row / G;
    const bool row_valid = tok < q_len;
    const int qpos = seq_len - q_len + tok;
    const int vis_end = p.causal ? min(qpos + 1, seq_len) : seq_len;
    const int vis_start = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
    const bool capped = p.softcap_log2 > 0.f;
    const float c = p.scale_log2;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + col_s(t);
    const uint32_t o_col = lane_base + col_o(t);
    // a sink logit starts the running state: it joins the denominator and adds no value
    float m_run = p.sinks != nullptr ? p.sinks[kvh * G + row % G] * kLog2e : -INFINITY;
    float l_run = p.sinks != nullptr ? 1.f : 0.f;
    bool ok = true;
    for (int j = 0; j < n_mine; ++j) {
      if (!warp_wait(&bars[B_SF + t], j & 1, abort_flag)) {
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
        rescale = (j > 0);
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
      // S_t(j) has landed, so P.V of tile j-1 (issued before it) is complete: O is stable
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
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
    if (ok && n_mine > 0 && !warp_wait(&bars[B_OD + t], (n_mine - 1) & 1, abort_flag)) ok = false;
    if (!ok) {
      set_abort(abort_flag, p.err);
    } else if (kPrefix) {
      // cascade prefix pass: the row's unnormalised partial (acc, m in log2 units, l) in the
      // split-partial layout the combine merges. (A tile without keys here has no valid rows:
      // ranges past the prefix end left the kernel at the top.)
      const size_t slot = ((size_t)(q_start + tok) * p.slot_count + r) * p.num_q_heads + kvh * G + row % G;
      float* acc = p.ws_acc + slot * kD;
      if (n_mine > 0) {
        tc_fence_after();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t ov[32];
          tmem_ld32(o_col + 32 * q4, ov);
          tmem_ld_wait();
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<uint4*>(acc + q4 * 32 + i) = make_uint4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
          }
        }
        if (row_valid) {
          p.ws_ml[slot * 2] = m_run;
          p.ws_ml[slot * 2 + 1] = l_run;
        }
      }
    } else if (n_mine > 0) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(q_start + tok) * p.out_stride +
                           (size_t)(kvh * G + row % G) * kD;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        tmem_ld32(o_col + 32 * q4, ov);
        tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[i + 4]) * inv, __uint_as_float(ov[i + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[i + 6]) * inv, __uint_as_float(ov[i + 7]) * inv);
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
      const int issued = *issued_tiles;
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        (void)mbar_wait(&bars[B_KF + j % kStages], (j / kStages) & 1);
        (void)mbar_wait(&bars[B_VF + j % kStages], (j / kStages) & 1);
      }
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
  return head_dim == kD && g_ok && bs_ok;
}

int varlen_tc_tokens_per_cta(int group) { return 2 * (kBM / group); }

cudaError_t launch_varlen_tc(const VarlenParams& p_in, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  VarlenParams p = p_in;
  if (p.out_stride == 0) p.out_stride = (long long)p.num_q_heads * kD;  // dense rows
  // the shared-memory opt-in is per device and kernel; setting it twice is harmless
  static std::atomic<bool> attr_done[64][2] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int mode = p.prefix_mode ? 1 : 0;
  auto kern = p.prefix_mode ? varlen_tc_kernel<true> : varlen_tc_kernel<false>;
  if (dev < 0 || dev >= 64 || !attr_done[dev][mode].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev][mode].store(true, std::memory_order_release);
  }
  const long long ctas = (p.work_items != nullptr && !p.prefix_mode ? (long long)p.num_items
                                                                     : (long long)p.q_tiles * p.num_reqs) *
                         p.num_kv_heads;
  if (ctas <= 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(p, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace pa
