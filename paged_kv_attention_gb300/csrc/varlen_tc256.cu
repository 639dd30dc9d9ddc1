// Varlen causal paged attention at head_dim 256 on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// The method is that of the head_dim 64/128 kernel ("32. Production attention kernels", One kernel
// for the whole batch; "TileInfer.jl - Attention kernels", Prefill): 128 packed GQA rows per query
// tile, query t of a request at seq_len - q_len + t, causal by position, FlashAttention-2 online
// softmax in fp32 with exp2, probabilities rounded to bf16 for P.V.
//
// What changes at head_dim 256 is the budget. A query tile is 64 KiB of shared memory and its
// output accumulator 256 TMEM columns, so two tiles (and their two score blocks) no longer fit
// the SM's 512 columns. This kernel therefore works on one query tile at a time (a CTA still owns
// the same two consecutive tiles of a (request, KV head) as the other kernel, A then B, so the
// work list and grid are the same) and overlaps its own softmax with the tensor core instead:
//  * TMEM: two score blocks S0, S1 (128 columns each) and O (256 columns). S(j + 1) is issued
//    into the other block as soon as its keys have landed, so the tensor core computes the next
//    scores while the softmax of tile j runs; the MMA order is S(0), S(1), PV(0), S(2), PV(1), ...;
//  * K and V arrive as half tiles (128 keys x 128 dims, 32 KiB) in one five-slot ring, in the
//    order the MMAs consume them: K(0) lo/hi, K(1) lo/hi, V(0) lo/hi, K(2) lo/hi, V(1) lo/hi, ...
//    (Q 64 KiB + ring 160 KiB fill the 227 KiB a CTA may use);
//  * S = Q K^T is 16 MMAs of M=128 N=128 K=16 (the first 8 read the low half of K, the next 8 the
//    high half); O += P V is 8 key steps x two N=128 MMAs, one per half of V, with P read from TMEM;
//  * warps 0-3 run the softmax (one thread per row), warp 4 is the producer (lane k copies page k
//    of a half tile), warp 5 the MMA issuer (one lane) and the V-tail zeroing (whole warp).
// O is rescaled in TMEM only when the running max rose by more than 2^8 (as in the other kernel);
// since PV(j-1) may still run when the softmax of tile j starts, that rescale first waits for it.
// Every wait is bounded; on expiry the CTA flags PA_ERRBIT_WAIT_TIMEOUT, drains its copies and
// MMAs, frees its tensor memory and exits.
#include <atomic>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kBM = 128;                 // packed query rows per tile
constexpr int kD = 256;                  // head dim of this kernel
constexpr int kRegion = 128 * 128;       // [128 rows][64 bf16] swizzled 64-column block: 16 KiB
constexpr int kHalfBytes = 2 * kRegion;  // 128 keys x 128 dims
constexpr int kSlots = 5;                // half-tile ring
constexpr int kOffQ = 0;                 // 4 blocks of 64 columns: 64 KiB
constexpr int kOffRing = kOffQ + 4 * kRegion;
constexpr int kOffBar = kOffRing + kSlots * kHalfBytes;
enum {
  B_FULL = 0,              // +slot: a half tile has landed
  B_EMPTY = B_FULL + kSlots,  // +slot: the MMAs that read it are done
  B_QF = B_EMPTY + kSlots,    // the query tile has landed (phase = tile 0, 1)
  B_QE,                       // the first tile's last S is done: the query buffer may be refilled
  B_SF,                       // +block (2): S(j) has landed in block j % 2
  B_PR = B_SF + 2,            // +block (2): P(j) is in block j % 2 (128 arrivals)
  B_OD = B_PR + 2,            // PV(j) is done (every PV, in order)
  B_OF,                       // the tile's last PV is done (phase = tile 0, 1)
  B_FIN,                      // drain after an abort
  kNumBars
};
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 32;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
__host__ __device__ constexpr uint32_t col_s(int b) { return b == 0 ? 0u : 128u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

// One query tile's schedule: its key tiles j0 .. j0 + n - 1 and where its counters start.
struct TileRun {
  int n_tok;   // valid tokens (0 = no such tile)
  int tok0;    // first token (within the request)
  int first;   // position of its first query
  int j0;      // first key tile
  int n;       // key tiles
  int s_base;  // index of its S(0) among the CTA's S operations
  int it_base; // index of its first ring item
};

// The MMAs consume ring items in the order S(0) [K(0) lo, hi], then for j = 1 .. n-1 S(j) [K(j)]
// and PV(j-1) [V(j-1)], then PV(n-1) [V(n-1)]. Item 2*op + h is half h of operation op.
// Operation op of a tile with n key tiles: (is_v, key tile).
__device__ __forceinline__ void op_of(int op, int n, bool& is_v, int& j) {
  if (op == 0) {
    is_v = false;
    j = 0;
  } else if (op == 2 * n - 1) {
    is_v = true;
    j = n - 1;
  } else {
    is_v = (op & 1) == 0;  // op 2k-1: S(k), op 2k: PV(k-1)
    j = is_v ? op / 2 - 1 : (op + 1) / 2;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    varlen_tc256_kernel(const __grid_constant__ VarlenParams p, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_items = reinterpret_cast<int*>(tmem_slot + 2);
  int* issued_q = reinterpret_cast<int*>(tmem_slot + 3);

  // ---- which tile pair: from the caller's plan, else heaviest (last) tile pairs first
  int tile, r, kvh;
  if (p.work_items != nullptr) {
    // a list planned on the device by the kernel launched just before this one: wait for it
    if (p.plan_on_device) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int item = p.plan_on_device ? p.work_items[blockIdx.x / p.num_kv_heads]
                                      : __ldg(p.work_items + blockIdx.x / p.num_kv_heads);
    kvh = (int)(blockIdx.x % p.num_kv_heads);
    if (item < 0) return;  // padding past the plan's last item
    tile = item / p.num_reqs;
    r = item - tile * p.num_reqs;
    if (tile >= p.q_tiles) {
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
  const int TOK = kBM / G;
  const int tid = threadIdx.x;
  const int q_start = p.query_start_loc[r];
  const int q_stop = p.query_start_loc[r + 1];
  const int seq_len = p.seq_lens[r];
  if (q_start >= 0 && q_stop <= p.num_tokens && q_stop - q_start >= 1 && q_stop - q_start <= p.skip_upto) return;
  const int q_len = q_stop - q_start;
  const bool layout_ok = q_start >= 0 && q_len >= 0 && q_stop <= p.num_tokens;
  const bool too_long = seq_len > p.max_blocks * p.block_size;
  const bool bad = !layout_ok || q_len > seq_len || too_long;
  const int tok0 = tile * 2 * TOK;
  if (bad) {
    if (tid == 0 && kvh == 0 && tile == 0)
      flag_error(p.err, too_long && layout_ok && q_len <= seq_len ? PA_ERRBIT_LENGTH_OUT_OF_RANGE
                                                                   : PA_ERRBIT_QUERY_LAYOUT);
    if (!layout_ok || tok0 >= q_len) return;
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
  if (tok0 >= q_len) return;

  // the CTA's two query tiles, A then B
  TileRun run[2];
  int n_items = 0, n_s = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const TileSpan sp = tile_span(tok0 + t * TOK, TOK, q_len, seq_len, p.causal);
    TileRun& u = run[t];
    u.n_tok = sp.n_tok;
    u.tok0 = tok0 + t * TOK;
    u.first = sp.first;
    u.j0 = (sp.n_tok > 0 && p.window > 0) ? max(0, sp.first - p.window + 1) / kBN : 0;
    u.n = sp.n_tok > 0 ? max(0, sp.n_kv - u.j0) : 0;
    u.s_base = n_s;
    u.it_base = n_items;
    n_s += u.n;
    n_items += 4 * u.n;
  }
  const int n_tiles = run[1].n > 0 ? 2 : 1;  // tile A always has keys (its first query sees key 0..)
  const int bs = p.block_size;
  const int pages_per_tile = kBN / bs;
  const int seq_pages = (seq_len + bs - 1) / bs;

  const int warp = tid >> 5, lane = tid & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars[B_FULL + s], 1);
      mbar_init(&bars[B_EMPTY + s], 1);
    }
    mbar_init(&bars[B_QF], 1);
    mbar_init(&bars[B_QE], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_SF + b], 1);
      mbar_init(&bars[B_PR + b], kBM);
    }
    mbar_init(&bars[B_OD], 1);
    mbar_init(&bars[B_OF], 1);
    mbar_init(&bars[B_FIN], 1);
    fence_barrier_init();
    *abort_flag = 0;
    *issued_items = 0;
    *issued_q = 0;
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

  if (warp == 4) {
    // ------------------------------------------------ producer: per tile its query, then the ring
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
    }
    const int32_t* table = p.block_tables + (size_t)r * p.max_blocks;
    int it = 0;
    bool ok = true;
    for (int t = 0; ok && t < n_tiles; ++t) {
      const TileRun& u = run[t];
      if (t == 1 && !warp_wait(&bars[B_QE], 0, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[B_QF], 4 * kRegion);
        for (int a = 0; a < 4; ++a)
          tma_load_3d(smem + kOffQ + a * kRegion, &qmap, &bars[B_QF], a * 64, kvh * G, q_start + u.tok0);
        *issued_q = t + 1;
      }
      for (int op = 0; op < 2 * u.n; ++op) {
        bool is_v;
        int j;
        op_of(op, u.n, is_v, j);
        const int jt = u.j0 + j;
        const int pg_idx = jt * pages_per_tile + lane;
        const int page = (lane < pages_per_tile && pg_idx < seq_pages) ? __ldg(table + pg_idx) : 0;
        const int p0 = jt * pages_per_tile;
        const int np = min(p0 + pages_per_tile, seq_pages) - p0;
        const uint32_t bytes = (uint32_t)np * bs * 256u;  // 128 dims of bf16 per key
        for (int h = 0; h < 2; ++h, ++it) {
          const int slot = it % kSlots;
          if (it >= kSlots && !warp_wait(&bars[B_EMPTY + slot], ((it / kSlots) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bars[B_FULL + slot], bytes);
          __syncwarp();
          if (lane < np) {
            if (page < 0 || page >= p.num_blocks) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // reads zeros
            uint8_t* dst = smem + kOffRing + slot * kHalfBytes + lane * bs * 128;
            for (int a = 0; a < 2; ++a)
              tma_load_4d(dst + a * kRegion, is_v ? &vmap : &kmap, &bars[B_FULL + slot], h * 128 + a * 64, kvh, 0,
                          page);
          }
          __syncwarp();
          if (lane == 0) *issued_items = it + 1;
        }
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) set_abort(abort_flag, p.err);
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer (lane 0); the warp zeroes V tails
    const uint32_t id_s = idesc_bf16(kBM, kBN, false);
    const uint32_t id_pv = idesc_bf16(kBM, 128, true);
    const uint64_t dq0 = sdesc(smem_addr(smem + kOffQ), 16, 1024);
    const uint64_t dring_k = sdesc(smem_addr(smem + kOffRing), 16, 1024);
    const uint64_t dring_v = sdesc(smem_addr(smem + kOffRing), kRegion, 1024);  // MN-major V
    bool ok = true;
    int it = 0;
    // release a slot to the producer only if it will refill it (an arrive nobody waits for could
    // land after this CTA has left)
    auto release = [&](int item) {
      if (lane == 0 && item + kSlots < n_items) umma_commit(&bars[B_EMPTY + item % kSlots]);
    };
    for (int t = 0; ok && t < n_tiles; ++t) {
      const TileRun& u = run[t];
      if (!(ok = warp_wait(&bars[B_QF], t & 1, abort_flag))) break;
      for (int op = 0; op < 2 * u.n; ++op, it += 2) {
        bool is_v;
        int j;
        op_of(op, u.n, is_v, j);
        const int sidx = u.s_base + j;  // S(j)'s index among the CTA's S operations
        const int blk = sidx & 1;
        if (is_v && !(ok = warp_wait(&bars[B_PR + blk], (sidx >> 1) & 1, abort_flag))) break;
        if (!(ok = warp_wait(&bars[B_FULL + it % kSlots], (it / kSlots) & 1, abort_flag))) break;
        if (!(ok = warp_wait(&bars[B_FULL + (it + 1) % kSlots], ((it + 1) / kSlots) & 1, abort_flag))) break;
        if (is_v) {
          // V rows at or past the sequence end: exact zeros (a stale slot may hold NaN)
          const int zero_from = seq_len - (u.j0 + j) * kBN;
          if (zero_from < kBN) {
            const int rows = kBN - zero_from;
            for (int h = 0; h < 2; ++h) {
              uint8_t* vbp = smem + kOffRing + ((it + h) % kSlots) * kHalfBytes;
              for (int i = lane; i < rows * 16; i += 32) {
                const int row = zero_from + i / 16, c = i % 16;
                *reinterpret_cast<uint4*>(vbp + (c >> 3) * kRegion + row * 128 + (c & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
            }
            fence_async_smem();
            __syncwarp();
          }
        }
        tc_fence_after();
        if (lane == 0) {
          if (!is_v) {
            // S(j) = Q K(j)^T into block blk: K steps 0-7 from the low half of K, 8-15 from the high.
            // Each half's slot is released as soon as the MMAs that read it are done, so the
            // producer can refill the low half's slot while the high half is still being read.
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const int half = kk >> 3;
              const uint64_t dk = dring_k + (uint64_t)((((it + half) % kSlots) * kHalfBytes) >> 4);
              const uint64_t offq = (uint64_t)(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
              const uint64_t offk = (uint64_t)((((kk >> 2) & 1) * kRegion + (kk & 3) * 32) >> 4);
              umma_ss(tmem + col_s(blk), dq0 + offq, dk + offk, id_s, kk > 0 ? 1u : 0u);
              if (kk == 7) release(it);
            }
            umma_commit(&bars[B_SF + blk]);
            release(it + 1);
            // the first tile's last S: the query buffer may be refilled with the second tile's
            if (t == 0 && n_tiles == 2 && j == u.n - 1) umma_commit(&bars[B_QE]);
          } else {
            // O += P(j) V(j): all 8 key steps of the low half of V (output columns 0-127), then of
            // the high half, each half's slot released once its MMAs are done
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk) {
                const uint64_t dv = dring_v + (uint64_t)((((it + h) % kSlots) * kHalfBytes + kk * 2048) >> 4);
                umma_ts(tmem + kColO + h * 128, tmem + col_s(blk) + 8 * kk, dv, id_pv,
                        (j > 0 || kk > 0) ? 1u : 0u);
              }
              if (h == 0) release(it);
            }
            umma_commit(&bars[B_OD]);
            if (j == u.n - 1) umma_commit(&bars[B_OF]);
            release(it + 1);
          }
        }
        __syncwarp();
      }
    }
    if (!ok) set_abort(abort_flag, p.err);
  } else {
    // ------------------------------------------------ softmax: warps 0-3, one thread per row
    const int row = tid & (kBM - 1);
    const bool capped = p.softcap_log2 > 0.f;
    const float c = p.scale_log2;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t o_col = lane_base + kColO;
    bool ok = true;
    for (int t = 0; ok && t < n_tiles; ++t) {
      const TileRun& u = run[t];
      const int tok = u.tok0 + row / G;
      const bool row_valid = tok < q_len;
      const int qpos = seq_len - q_len + tok;
      const int vis_end = p.causal ? min(qpos + 1, seq_len) : seq_len;
      const int vis_start = p.window > 0 ? max(0, qpos - p.window + 1) : 0;
      float m_run = p.sinks != nullptr ? p.sinks[kvh * G + row % G] * kLog2e : -INFINITY;
      float l_run = p.sinks != nullptr ? 1.f : 0.f;
      for (int j = 0; j < u.n; ++j) {
        const int sidx = u.s_base + j;
        const int blk = sidx & 1;
        const uint32_t s_col = lane_base + col_s(blk);
        if (!warp_wait(&bars[B_SF + blk], (sidx >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nvis = vis_end - (u.j0 + j) * kBN;
        const int nlo = vis_start - (u.j0 + j) * kBN;
        const bool full = nvis >= kBN && nlo <= 0;
        uint32_t sv[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(s_col + 32 * q4, sv[q4]);
        tmem_ld_wait();
        if (!full) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sv[q4][i] = (q4 * 32 + i < nvis && q4 * 32 + i >= nlo) ? sv[q4][i] : __float_as_uint(-INFINITY);
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sv[q4][i]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
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
            if (capped) {
              x0 = p.softcap_log2 * tanh_ex2(__uint_as_float(src[e]) * p.scale_over_cap) - mu;
              x1 = p.softcap_log2 * tanh_ex2(__uint_as_float(src[e + 1]) * p.scale_over_cap) - mu;
              x0 = __uint_as_float(src[e]) == -INFINITY ? -INFINITY : x0;
              x1 = __uint_as_float(src[e + 1]) == -INFINITY ? -INFINITY : x1;
            } else {
              f2_split(f2_fma(f2(__uint_as_float(src[e]), __uint_as_float(src[e + 1])), c2, nmu2), x0, x1);
            }
            const float p0 = ex2(x0), p1 = ex2(x1);
            sum2[i & 1] = f2_add(sum2[i & 1], f2(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st32(s_col + 32 * h, pk);
        }
        float la, lb;
        f2_split(f2_add(sum2[0], sum2[1]), la, lb);
        l_run = l_run * alpha + (la + lb);
        m_run = m_new;
        if (__any_sync(0xffffffffu, rescale)) {
          // PV(j-1) may still be accumulating into O (S(j) was issued before it): wait for it. Every
          // PV up to PV(j-2) is done (issued before S(j), which has landed) and PV(j) is not issued,
          // so the barrier is at most one phase behind and its parity wait cannot alias.
          const int od = run[t].s_base + j - 1;  // PV operations before PV(j-1) of this tile
          if (!warp_wait(&bars[B_OD], od & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
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
        mbar_arrive(&bars[B_PR + blk]);
      }
      if (!ok) break;
      if (!warp_wait(&bars[B_OF], t & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)(q_start + tok) * p.out_stride +
                           (size_t)(kvh * G + row % G) * kD;
#pragma unroll
      for (int q4 = 0; q4 < kD / 32; ++q4) {
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
      // the next tile's first PV overwrites O: it is issued only after this warp's P-ready arrive,
      // which follows these loads in program order
      tc_fence_before();
    }
    if (!ok) set_abort(abort_flag, p.err);
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
      // the second query load is issued only after the first one landed, so the last suffices
      const int nq = *issued_q;
      if (nq > 0) (void)mbar_wait(&bars[B_QF], (nq - 1) & 1);
      const int issued = *issued_items;
      for (int i = max(0, issued - kSlots); i < issued; ++i)
        (void)mbar_wait(&bars[B_FULL + i % kSlots], (i / kSlots) & 1);
    }
    __syncthreads();
  }
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

cudaError_t launch_varlen_tc256(const VarlenParams& p, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, long long ctas, cudaStream_t stream) {
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(varlen_tc256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  if (!p.plan_on_device) {
    varlen_tc256_kernel<<<(unsigned)ctas, kThreads, kSmemBytes, stream>>>(p, qmap, kmap, vmap);
    return cudaGetLastError();
  }
  return launch_dependent(varlen_tc256_kernel, (unsigned)ctas, kThreads, kSmemBytes, stream, p, qmap, kmap, vmap);
}

}  // namespace pa
