// Varlen causal paged attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Method ("32. Production attention kernels", One kernel for the whole batch;
// "TileInfer.jl - Attention kernels", Prefill and Walking the block table):
//  * one CTA per (query tile, request, KV head). A query tile is 128 packed rows: 128/G
//    consecutive query tokens of the request times the G query heads of the KV head
//    (row m = token m / G, head m % G), so each K/V tile serves the whole group;
//  * request r's q_len queries are the newest of its seq_len positions (query t sits at
//    seq_len - q_len + t) and see keys up to their own position; the key loop stops at the
//    tile's last query and only tiles that cross the diagonal or the sequence end are masked;
//  * FlashAttention-2 online softmax in fp32 with exp2 (scale pre-multiplied by log2 e);
//    probabilities are rounded to bf16 for the P.V product.
//
// GB300 mapping:
//  * warp 4 (one lane) walks the block table and issues TMA loads: the Q tile once, then a
//    two-stage ring of 128-key K and V tiles, one box per page per 64-column half, in the
//    128-byte-swizzled layout the tensor core reads directly;
//  * warp 5 owns the tensor memory (512 columns: two 128-column score buffers and the
//    128-column output accumulator) and one lane issues tcgen05.mma: S = Q K^T (M=128,
//    N=128, K=128) into the free score buffer while the softmax works on the other, then
//    O += P V (two N=64 halves) once the softmax has written P;
//  * warps 0-3 (one thread per row) read S from TMEM, mask, update the running max/sum,
//    write P (bf16, swizzled) to shared memory and rescale O in TMEM only when the running
//    max rose by more than 2^8 (the result is exact for any reference max; this only
//    bounds the fp32 range of P and O);
//  * every wait is bounded; on expiry the CTA flags PA_ERRBIT_WAIT_TIMEOUT, drains its
//    outstanding copies and MMAs, frees its tensor memory and exits.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kBM = 128;  // packed query rows per tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kD = 128;   // head dim of this kernel
constexpr int kStages = 2;
constexpr int kRegion = 128 * 128;      // one [128 rows][64 bf16] swizzled column half: 16 KiB
constexpr int kTileBytes = 2 * kRegion; // a 128 x 128 bf16 tile
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
enum { B_Q = 0, B_KF = 1, B_VF = 3, B_KVE = 5, B_SF = 7, B_P = 9, B_O = 10, B_FIN = 11, kNumBars = 12 };
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 32;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
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

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
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

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
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

__global__ void __launch_bounds__(kThreads, 1)
    varlen_tc_kernel(const __grid_constant__ VarlenParams p, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_tiles = reinterpret_cast<int*>(tmem_slot + 2);

  // ---- which tile: heaviest (last) query tiles first across all requests and heads
  const int per_tile = p.num_reqs * p.num_kv_heads;
  const int tile = p.q_tiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int r = rem / p.num_kv_heads;
  const int kvh = rem - r * p.num_kv_heads;
  const int G = p.group;
  const int TOK = kBM / G;
  const int tid = threadIdx.x;

  const int q_start = p.query_start_loc[r];
  const int q_stop = p.query_start_loc[r + 1];
  const int seq_len = p.seq_lens[r];
  const int q_len = q_stop - q_start;
  const bool layout_ok = q_start >= 0 && q_len >= 0 && q_stop <= p.num_tokens;
  const bool too_long = seq_len > p.max_blocks * p.block_size;
  const bool bad = !layout_ok || q_len > seq_len || too_long;
  if (bad) {
    if (tid == 0 && kvh == 0 && tile == 0)
      flag_error(p.err, too_long && layout_ok && q_len <= seq_len ? PA_ERRBIT_LENGTH_OUT_OF_RANGE
                                                                   : PA_ERRBIT_QUERY_LAYOUT);
    if (!layout_ok) return;
    // a request the kernel cannot serve gives zero rows
    const int tok0 = tile * TOK;
    if (tok0 >= q_len) return;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    const int rows = min(TOK, q_len - tok0) * G;
    for (int i = tid; i < rows * (kD / 8); i += blockDim.x) {
      const int row = i / (kD / 8), c = i % (kD / 8);
      const size_t o = ((size_t)(q_start + tok0 + row / G) * p.num_q_heads + kvh * G + row % G) * kD + c * 8;
      *reinterpret_cast<uint4*>(out + o) = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  if (tile == 0 && kvh == 0 && tid == 0 && q_len > p.max_query_len) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
  const int tok0 = tile * TOK;
  if (tok0 >= q_len) return;  // nothing of this request in this tile (uniform: whole CTA leaves)

  const int n_tok = min(TOK, q_len - tok0);
  const int first_pos = seq_len - q_len + tok0;
  const int key_end = p.causal ? min(seq_len, first_pos + n_tok) : seq_len;  // keys [0, key_end)
  const int n_kv = (key_end + kBN - 1) / kBN;
  const int bs = p.block_size;
  const int pages_per_tile = kBN / bs;
  const int seq_pages = (seq_len + bs - 1) / bs;

  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_KF + s], 1);
      mbar_init(&bars[B_VF + s], 1);
      mbar_init(&bars[B_KVE + s], 1);
      mbar_init(&bars[B_SF + s], 1);
    }
    mbar_init(&bars[B_P], kBM);
    mbar_init(&bars[B_O], 1);
    mbar_init(&bars[B_FIN], 1);
    fence_barrier_init();
    *abort_flag = 0;
    *issued_tiles = 0;
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = smem_addr(smem + kOffQ);
  const uint32_t sK = smem_addr(smem + kOffK);
  const uint32_t sV = smem_addr(smem + kOffV);
  const uint32_t sP = smem_addr(smem + kOffP);

  if (warp == 4) {
    // ------------------------------------------------ producer: Q once, then K/V tiles
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      mbar_arrive_expect_tx(&bars[B_Q], kTileBytes);
      for (int a = 0; a < 2; ++a)
        tma_load_3d(smem + kOffQ + a * kRegion, &qmap, &bars[B_Q], a * 64, kvh * G, q_start + tok0);
      const int32_t* table = p.block_tables + (size_t)r * p.max_blocks;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        if (j >= kStages && !wait_or_abort(&bars[B_KVE + st], ((j / kStages) - 1) & 1, abort_flag)) {
          set_abort(abort_flag, p.err);
          break;
        }
        const int p0 = j * pages_per_tile;
        const int p1 = min(p0 + pages_per_tile, seq_pages);
        const uint32_t bytes = (uint32_t)(p1 - p0) * bs * 256u;
        mbar_arrive_expect_tx(&bars[B_KF + st], bytes);
        for (int pg = p0; pg < p1; ++pg) {
          const int page = table[pg];
          if (page < 0 || page >= p.num_blocks) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // reads zeros
          for (int a = 0; a < 2; ++a)
            tma_load_4d(smem + kOffK + st * kTileBytes + a * kRegion + (pg - p0) * bs * 128, &kmap,
                        &bars[B_KF + st], a * 64, kvh, 0, page);
        }
        mbar_arrive_expect_tx(&bars[B_VF + st], bytes);
        for (int pg = p0; pg < p1; ++pg) {
          const int page = table[pg];
          for (int a = 0; a < 2; ++a)
            tma_load_4d(smem + kOffV + st * kTileBytes + a * kRegion + (pg - p0) * bs * 128, &vmap,
                        &bars[B_VF + st], a * 64, kvh, 0, page);
        }
        *issued_tiles = j + 1;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer (lane 0); the warp zeroes V tails
    const uint32_t id_s = idesc_bf16(kBM, kBN, false);
    const uint32_t id_pv = idesc_bf16(kBM, 64, true);
    bool ok = warp_wait(&bars[B_Q], 0, abort_flag);
    auto issue_s = [&](int j) -> bool {
      const int st = j % kStages;
      if (!warp_wait(&bars[B_KF + st], (j / kStages) & 1, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = tmem + (uint32_t)((j & 1) * kBN);
        const uint32_t kb = sK + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kRegion + (kk & 3) * 32;
          umma_bf16(d, sdesc(sQ + off, 16, 1024), sdesc(kb + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_SF + (j & 1)]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
      if (!(ok = warp_wait(&bars[B_P], j & 1, abort_flag))) break;
      const int st = j % kStages;
      if (!(ok = warp_wait(&bars[B_VF + st], (j / kStages) & 1, abort_flag))) break;
      const int zero_from = seq_len - j * kBN;  // V rows at or past the sequence end: exact zeros
      if (zero_from < kBN) {
        uint8_t* vb = smem + kOffV + st * kTileBytes;
        const int rows = kBN - zero_from;
        for (int i = lane; i < rows * 16; i += 32) {
          const int row = zero_from + i / 16, c = i % 16;
          *reinterpret_cast<uint4*>(vb + (c >> 3) * kRegion + row * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = sV + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t a = sdesc(sP + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            umma_bf16(tmem + kColO + 64 * h, a, sdesc(vb + h * kRegion + kk * 2048, 1024, 1024), id_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        // release the stage only when the producer will refill it: an arrive that nobody
        // waits for could land after this CTA has left
        if (j + kStages < n_kv) umma_commit(&bars[B_KVE + st]);
        umma_commit(&bars[B_O]);
      }
      __syncwarp();
    }
    if (!ok) set_abort(abort_flag, p.err);
  } else {
    // ------------------------------------------------ softmax: one thread per packed row
    const int row = tid;
    const int t = tok0 + row / G;
    const bool row_valid = t < q_len;
    const int qpos = seq_len - q_len + t;
    const int vis_end = p.causal ? min(qpos + 1, seq_len) : seq_len;
    const float c = p.scale_log2;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint8_t* prow = smem + kOffP + row * 128;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(&bars[B_SF + (j & 1)], (j >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(lane_base + (uint32_t)((j & 1) * kBN + 32 * q4), sv[q4]);
      tmem_ld_wait();
      const int nvis = vis_end - j * kBN;
      float mx = -INFINITY;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = __uint_as_float(sv[q4][i]);
          x = (q4 * 32 + i < nvis) ? x : -INFINITY;  // select: NaN past the end never survives
          sv[q4][i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      const float mxs = mx * c;
      float m_new = m_run, alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY || mxs > m_run + kRescaleThreshold) {
        m_new = mxs;
        alpha = exp2f(m_run - (m_new == -INFINITY ? 0.f : m_new));
        rescale = (j > 0);
      }
      const float mu = (m_new == -INFINITY) ? 0.f : m_new;
      float lsum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = exp2f(fmaf(__uint_as_float(sv[q4][i]), c, -mu));
          const float p1 = exp2f(fmaf(__uint_as_float(sv[q4][i + 1]), c, -mu));
          lsum += p0 + p1;
          pk[q4 * 16 + i / 2] = pack_bf16x2(p0, p1);
        }
      l_run = l_run * alpha + lsum;
      m_run = m_new;
      // P and O belong to the previous P.V until it completes
      if (j > 0 && !warp_wait(&bars[B_O], (j - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int region = u >> 3, unit = u & 7;
        *reinterpret_cast<uint4*>(prow + region * kRegion + ((unit ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kColO + 32 * q4, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
          tmem_st32(lane_base + kColO + 32 * q4, ov);
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_P]);
    }
    if (ok && !warp_wait(&bars[B_O], (n_kv - 1) & 1, abort_flag)) ok = false;
    if (!ok) {
      set_abort(abort_flag, p.err);
    } else {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) +
                           ((size_t)(q_start + t) * p.num_q_heads + kvh * G + row % G) * kD;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + 32 * q4, ov);
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
    if (warp == 5 && lane == 0) {
      umma_commit(&bars[B_FIN]);
      (void)mbar_wait(&bars[B_FIN], 0);
    }
    if (warp == 4 && lane == 0) {
      (void)mbar_wait(&bars[B_Q], 0);
      const int issued = *issued_tiles;
      for (int j = max(0, issued - kStages); j < issued; ++j) {
        (void)mbar_wait(&bars[B_KF + j % kStages], (j / kStages) & 1);
        (void)mbar_wait(&bars[B_VF + j % kStages], (j / kStages) & 1);
      }
    }
    __syncthreads();
  }
  if (warp == 5) {
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

cudaError_t launch_varlen_tc(const VarlenParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(varlen_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long ctas = (long long)p.q_tiles * p.num_reqs * p.num_kv_heads;
  if (ctas <= 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  varlen_tc_kernel<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(p, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace pa
