// Split-KV paged decode for sm_103a, and the log-sum-exp combine.
//
// Method ("TileInfer.jl - Attention kernels", Decode: GQA packing and split-KV;
// "32. Production attention kernels", Long contexts: split the keys):
//  * one CTA per (unit, KV head, split); the query heads that share the KV head form the
//    rows of one query tile, so every page of keys and values is read from HBM once per
//    group (a unit of several queries, a short varlen request, stacks their groups: rows =
//    queries x group, each row masked to its own query's causal range);
//  * the CTA walks its share of the block table 16 tokens at a time: a producer warp reads
//    the page id (a scalar load) and issues TMA loads of that page's rows for this KV head
//    into a ring of shared-memory stages;
//  * consumer warps take stages in turn and run the FlashAttention-2 online softmax with
//    fp32 scores in the exp2 domain (scale pre-multiplied by log2 e);
//  * a split writes its unnormalised partial (acc, m, l) to an fp32 workspace, or the
//    normalised output directly when there is one split; empty splits write the neutral
//    partial (0, -inf, 0) by the same arithmetic.
//
// bf16 path: the score and P.V products run on the tensor cores as mma.sync m16n8k16 with
// keys on M (16 per stage) and the packed query rows on N (8 per tile, two tiles for
// groups of 9-16). Decode does about 4 flops per byte of cache, so the tensor pipe is far
// from the limit; the point of the MMA is to keep the issue slots free for the memory
// pipeline. The probabilities are moved from the score accumulator layout to the P.V
// operand layout with movmatrix (an in-register 8x8 transpose), without shared memory.
#include <atomic>

#include "decode_common.cuh"

namespace pa {
namespace {

using namespace dec;

template <int D, int NT, int QK>
__global__ void __launch_bounds__(DecCfg<D, QK>::kThreads)
    decode_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
  using C = DecCfg<D, QK>;
  constexpr int ROWS = 8 * NT;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms must start on 1024-byte boundaries of the shared window
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty = full + C::kStages;
  float* merge_ml = reinterpret_cast<float*>(empty + C::kStages);  // [consumers][ROWS][2]
  float* scales = merge_ml + C::kConsumers * 16 * 2;                // [stages][32] (8-bit caches)
  float* merge_o = reinterpret_cast<float*>(smem);                 // aliases the ring after the loop
  __shared__ int s_timeout;
  __shared__ int s_issued[C::kProducers];

  const int unit = blockIdx.x / p.num_splits;
  const int split = blockIdx.x - unit * p.num_splits;
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Decode and request units: the block-table row follows from the unit alone, and this split's
  // first page is known before its length is, so the producer starts its first page-id window
  // load now and the two memory latencies overlap. (A window that turns out to start later than
  // the split is simply reloaded.)
  int spec_base = -64, spec_page = -1;
  if (warp >= C::kConsumers && lane == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (p.varlen != 1 && warp >= C::kConsumers) {
    // the unit's block-table row: the sequence, or (request units) the request of the group
    const int spec_row = p.varlen == 2 ? unit / p.groups_per_req : unit;
    spec_base = split * p.chunks_per_split * kChunk / p.block_size;
    spec_page = spec_base + lane < p.max_blocks
                    ? __ldg(p.block_tables + (size_t)spec_row * p.max_blocks + spec_base + lane)
                    : -1;
  }
  const Unit u = resolve_unit(p, unit, threadIdx.x == 0 && split == 0 && kvh == 0);
  // Launched to overlap the previous kernel on the stream (which this one does not read): one CTA
  // waits for that kernel's completion before it exits, so this grid completes only after it and
  // a kernel that waits for this grid also sees the previous one's writes. (A no-op otherwise.)
  const bool waits_for_previous = p.overlap_previous && blockIdx.x == 0 && blockIdx.y == 0;
  if (u.skip) {  // uniform: another kernel serves this unit
    if (waits_for_previous) asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  const int n_chunks = (u.len + kChunk - 1) / kChunk;
  const int c_begin = max(split * p.chunks_per_split, u.start / kChunk);
  const int c_end = min(n_chunks, split * p.chunks_per_split + p.chunks_per_split);
  const int n_mine = max(0, c_end - c_begin);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      // 8-bit caches: the 32 scale copies of a stage arrive on its barrier too
      mbar_init(&full[i], QK != 0 ? 33 : 1);
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
    s_timeout = 0;
    for (int w = 0; w < C::kProducers; ++w) s_issued[w] = 0;
  }
  __syncthreads();

  if (warp >= C::kConsumers) {
    // ---------------- producer: page-table walk + TMA (and, for 8-bit caches, the scales)
    if (n_mine > 0) {
      const int32_t* table = p.block_tables + (size_t)u.table_row * p.max_blocks;
      // page ids are fetched 32 at a time, one per lane, and handed out by shuffle: one
      // table-load latency per 32 pages instead of one per chunk
      int win_base = spec_base, my_page = spec_page;
      const int pw = warp - C::kConsumers;
      int issued = 0;
      for (int i = pw; i < n_mine; i += C::kProducers) {
        const int stage = i % C::kStages;
        bool ok = true;
        if (i >= C::kStages) ok = mbar_wait(&empty[stage], ((i / C::kStages) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) {
            flag_error(p.err, PA_ERRBIT_WAIT_TIMEOUT);
            atomicExch(&s_timeout, 1);
          }
          break;
        }
        const int tok = (c_begin + i) * kChunk;
        const int page_idx = tok / p.block_size;
        const int in_page = tok - page_idx * p.block_size;
        if (page_idx - win_base >= 32) {  // uniform: every lane has the same page_idx
          win_base = page_idx;
          my_page = (win_base + lane < p.max_blocks) ? __ldg(table + win_base + lane) : -1;
        }
        const int page = __shfl_sync(0xffffffffu, my_page, page_idx - win_base);
        const bool page_ok = page >= 0 && page < p.num_blocks;
        if constexpr (QK != 0) {
          // lanes 0-15: the chunk's key scales, 16-31: its value scales, copied asynchronously
          // (the producer never waits on them); positions past the sequence end, or on a page
          // outside the pool, are zero-filled instead of read
          const int t = lane & 15;
          const bool take = page_ok && tok + t < u.len;
          const float* base = lane < 16 ? p.k_scales : p.v_scales;
          const float* src = take ? base + ((size_t)page * p.block_size + in_page + t) * p.num_kv_heads + kvh : base;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(scales + stage * 32 + lane)),
                       "l"(src), "r"(take ? 4 : 0)
                       : "memory");
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&full[stage]))
                       : "memory");
        }
        if (lane == 0) {
          if (!page_ok) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // TMA reads zeros
          uint8_t* st = smem + stage * C::kStageBytes;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          if constexpr (C::kBoxes > 1) {  // every 128-byte column of the chunk in one copy (5-D map)
            tma_load_5d(st, &kmap, &full[stage], 0, in_page, 0, kvh, page);
            tma_load_5d(st + C::kTileBytes, &vmap, &full[stage], 0, in_page, 0, kvh, page);
          } else {
            tma_load_4d(st, &kmap, &full[stage], 0, kvh, in_page, page);
            tma_load_4d(st + C::kTileBytes, &vmap, &full[stage], 0, kvh, in_page, page);
          }
        }
        issued = i + 1;
      }
      if (lane == 0) s_issued[pw] = issued;
    }
  } else {
    // ---------------- consumers
    const int G = p.group;
    const int g4 = lane >> 2;  // groupID
    const int t4 = lane & 3;   // thread in group
    // Q^T as the B operand: rows n = (query t = n / G of the unit, head n % G of the group),
    // k = head dim
    const int n_rows = u.n_tok * G;
    uint32_t qf[NT][C::kMT][2];
    {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + g4;
        const bool rv = n < n_rows;
        const int t = rv ? n / G : 0;
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const __nv_bfloat16*>(p.q) + (size_t)(u.q_row + t) * p.q_stride +
            (size_t)(kvh * G + (rv ? n - t * G : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < C::kMT; ++kk) {
          if constexpr (QK == 0) {
            qf[nt][kk][0] = rv ? __ldg(qr + (kk * 16 + 2 * t4) / 2) : 0u;
            qf[nt][kk][1] = rv ? __ldg(qr + (kk * 16 + 8 + 2 * t4) / 2) : 0u;
          } else {
            // the codes' k-slot order (dims 4t..4t+3 of each 16-dim step), converted to fp16
            qf[nt][kk][0] = rv ? bf16x2_to_f16x2(__ldg(qr + (kk * 16 + 4 * t4) / 2)) : 0u;
            qf[nt][kk][1] = rv ? bf16x2_to_f16x2(__ldg(qr + (kk * 16 + 4 * t4 + 2) / 2)) : 0u;
          }
        }
      }
    }
    // int8: 1152 times each score row's query dim sum (rows 2 t4 and 2 t4 + 1 of every 8), the
    // offset the biased key codes add to its scores; the sum is over the fp16 queries the MMAs use
    float qb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float part = 0.f;
      if constexpr (QK == 1) {
#pragma unroll
        for (int kk = 0; kk < C::kMT; ++kk) {
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qf[nt][kk][0]));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&qf[nt][kk][1]));
          part += (a.x + a.y) + (b.x + b.y);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);  // lanes 4n..4n+3 now hold row n's sum
      }
      qb[nt][0] = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * t4);
      qb[nt][1] = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * t4 + 4);
    }
    // the keys each of this thread's score rows (2 t4 and 2 t4 + 1 of every 8) may see: query t
    // of the unit sees positions [first_pos + t - window + 1, first_pos + t] when causal (all
    // len when not); a one-query unit's rows all see [start, len)
    int key_hi[NT][2], key_lo[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = nt * 8 + 2 * t4 + j;
        const int t = n < n_rows ? n / G : u.n_tok - 1;
        key_hi[nt][j] = p.causal ? u.len - (u.n_tok - 1 - t) : u.len;
        key_lo[nt][j] = p.window > 0 ? u.first_pos + t - p.window + 1 : 0;
      }
    // keys in [all_lo, all_hi) are visible to every row: chunks inside need no mask at all
    const int all_hi = p.causal ? u.len - (u.n_tok - 1) : u.len;
    const int all_lo = p.window > 0 ? u.first_pos + u.n_tok - p.window : 0;
    float o[NT][C::kMT][4];
    float m_run[NT][2], l_run[NT][2];
    float psum[NT][4];  // int8: the probability sums of P.V's columns (its offset is 1152 times them)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
      psum[nt][0] = psum[nt][1] = psum[nt][2] = psum[nt][3] = 0.f;
#pragma unroll
      for (int mt = 0; mt < C::kMT; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
    }
    const float sl2 = p.scale_log2;
    // ldmatrix lane addressing: matrix mi = lane/8 supplies row ri = lane%8
    const int mi = lane >> 3, ri = lane & 7;
    const int k_key = ri + 8 * (mi & 1), k_unit = mi >> 1;  // K: (keys 0-7|8-15) x (unit u0|u0+1)
    const int v_key = ri + 8 * (mi >> 1), v_unit = mi & 1;  // V^T: (d 0-7|8-15) x (keys 0-7|8-15)
    constexpr int kRegionStride = kChunk * 128;  // bytes between the 128-byte columns of a tile

    for (int i = warp; i < n_mine; i += C::kConsumers) {
      const int stage = i % C::kStages;
      if (!mbar_wait(&full[stage], (i / C::kStages) & 1)) {
        flag_error(p.err, PA_ERRBIT_WAIT_TIMEOUT);
        atomicExch(&s_timeout, 1);
        break;
      }
      uint8_t* kt = smem + stage * C::kStageBytes;
      uint8_t* vt = kt + C::kTileBytes;
      const int key0 = (c_begin + i) * kChunk;
      const int nvalid = min(kChunk, u.len - key0);
      float ks_a = 1.f, ks_b = 1.f, vs_a = 1.f, vs_b = 1.f;
      // 8-bit caches: the chunk's codes go to registers (per thread 16 bytes of K and of V per
      // 128 head dims) and the stage is released before any arithmetic; at D 256 the value codes
      // are loaded after the scores, which keeps the two sets from being live together
      uint32_t kw[QK ? C::kMT : 1][2], vw[QK ? C::kMT : 1][2];
      // ldmatrix of matrices (keys 0-7 | 8-15) x (16-byte units u0 | u0+1) of 32 head dims
      auto load_codes = [&](const uint8_t* tile, uint32_t (&w)[QK ? C::kMT : 1][2], bool trans) {
#pragma unroll
        for (int k2 = 0; k2 < C::kMT / 2; ++k2) {
          const uint32_t off = (k2 >> 2) * kRegionStride + swz128(k_key, 2 * (k2 & 3) + k_unit);
          uint32_t r[4];
          if (trans) ldsm_x4_trans(r, smem_addr(tile + off)); else ldsm_x4(r, smem_addr(tile + off));
          w[2 * k2][0] = r[0];
          w[2 * k2][1] = r[1];
          w[2 * k2 + 1][0] = r[2];
          w[2 * k2 + 1][1] = r[3];
        }
      };
      // value codes of keys past the sequence end (anything, NaN codes included) become 0, so
      // 0-probability keys contribute exactly 0 to P.V; this thread holds keys 2t, 2t+1 (bytes
      // 0-1, 2-3) of keys 0-7 and the same of keys 8-15
      auto load_values_and_release = [&]() {
        load_codes(vt, vw, true);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);  // the codes are in registers
        if (nvalid < kChunk) {
          const uint32_t m0 = (2 * t4 < nvalid ? 0x0000ffffu : 0u) | (2 * t4 + 1 < nvalid ? 0xffff0000u : 0u);
          const uint32_t m1 =
              (2 * t4 + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * t4 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt) {
            vw[mt][0] &= m0;
            vw[mt][1] &= m1;
          }
        }
      };
      constexpr bool kLateValues = QK != 0 && D > 128;
      if constexpr (QK != 0) {
        const float* sc = scales + stage * 32;
        ks_a = sc[g4];
        ks_b = sc[g4 + 8];
        vs_a = sc[16 + g4];
        vs_b = sc[16 + g4 + 8];
        load_codes(kt, kw, false);
        if constexpr (!kLateValues) load_values_and_release();
      } else if (nvalid < kChunk) {
        // rows past the sequence end may hold anything (NaN included): zero them so that
        // 0-probability keys contribute exactly 0 to P.V (a select, not a multiply)
        for (int idx = lane; idx < (kChunk - nvalid) * (D / 64) * 8; idx += 32) {
          const int row = nvalid + idx / ((D / 64) * 8);
          const int rest = idx % ((D / 64) * 8);
          reinterpret_cast<uint4*>(vt + (rest / 8) * (kChunk * 128) + row * 128)[rest % 8] = make_uint4(0, 0, 0, 0);
        }
        // these generic-proxy writes precede the next TMA write of this stage
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      // S^T[16 keys x 8 rows] = K . Q^T; for E4M3 caches in two accumulator chains (even and odd
      // 16-dim steps, summed after), which halves the dependent MMA chain of a chunk (for int8 the
      // four more registers cost more than the shorter chain gains)
      constexpr int kChains = QK == 2 ? 2 : 1;
      float s[NT][4], s2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
      }
#pragma unroll
      for (int kk = 0; kk < C::kMT; ++kk) {
        uint32_t a[4];
        if constexpr (QK == 0) {
          const int dch = kk >> 2;
          const int unit_idx = 2 * (kk & 3) + k_unit;
          ldsm_x4(a, smem_addr(kt + dch * kRegionStride + swz128(k_key, unit_idx)));
        } else if constexpr (QK == 1) {  // the same slots, biased codes
          const uint32_t w0 = kw[kk][0] ^ 0x80808080u, w1 = kw[kk][1] ^ 0x80808080u;
          a[0] = biased2_to_f16x2(w0, kSelB01);
          a[1] = biased2_to_f16x2(w1, kSelB01);
          a[2] = biased2_to_f16x2(w0, kSelB23);
          a[3] = biased2_to_f16x2(w1, kSelB23);
        } else {  // keys g, g+8 x k-slots (2t, 2t+1 | 2t+8, 2t+9) = dims (4t, 4t+1 | 4t+2, 4t+3)
          e4m3_halves_to_f16x2(kw[kk][0], a[0], a[2]);
          e4m3_halves_to_f16x2(kw[kk][1], a[1], a[3]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_cache<QK>(kChains == 2 && (kk & 1) ? s2[nt] : s[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
      }
      if constexpr (kChains == 2) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
      }
      if constexpr (kLateValues) load_values_and_release();
      // online softmax (rows 2*t4 and 2*t4+1; keys g4 and g4+8)
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if constexpr (QK == 1) {  // the biased keys' offset (columns 2 t4, 2 t4 + 1)
          s[nt][0] -= qb[nt][0];
          s[nt][1] -= qb[nt][1];
          s[nt][2] -= qb[nt][0];
          s[nt][3] -= qb[nt][1];
        }
        if constexpr (QK != 0) {  // a key's scale multiplies its scores
          s[nt][0] *= ks_a;
          s[nt][1] *= ks_a;
          s[nt][2] *= ks_b;
          s[nt][3] *= ks_b;
        }
        float x0, x1, x2, x3;
        if (p.softcap_log2 > 0.f) {
          x0 = score_log2(p, s[nt][0]);
          x1 = score_log2(p, s[nt][1]);
          x2 = score_log2(p, s[nt][2]);
          x3 = score_log2(p, s[nt][3]);
        } else {
          x0 = s[nt][0] * sl2, x1 = s[nt][1] * sl2, x2 = s[nt][2] * sl2, x3 = s[nt][3] * sl2;
        }
        if (key0 + kChunk > all_hi || key0 < all_lo) {  // uniform: the sequence's ends only
          const int ka = key0 + g4, kb = ka + 8;  // positions of this thread's two keys
          if (ka >= key_hi[nt][0] || ka < key_lo[nt][0]) x0 = -INFINITY;
          if (ka >= key_hi[nt][1] || ka < key_lo[nt][1]) x1 = -INFINITY;
          if (kb >= key_hi[nt][0] || kb < key_lo[nt][0]) x2 = -INFINITY;
          if (kb >= key_hi[nt][1] || kb < key_lo[nt][1]) x3 = -INFINITY;
        }
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // lazy rescaling: a row's reference maximum moves only when a score passes it by more
        // than 2^8 (log2 units), so most chunks skip the accumulator rescale; (acc, m, l) stay
        // consistent with whichever reference is kept, and probabilities stay below 2^8. The
        // decision is the same in the 8 threads of a row (they share the row maximum).
        const bool up0 = mx0 > m_run[nt][0] + kLazyRescale, up1 = mx1 > m_run[nt][1] + kLazyRescale;
        const float mn0 = up0 ? mx0 : m_run[nt][0], mn1 = up1 ? mx1 : m_run[nt][1];
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0, mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float p0 = ex2_ftz(x0 - mu0), p2 = ex2_ftz(x2 - mu0);
        const float p1 = ex2_ftz(x1 - mu1), p3 = ex2_ftz(x3 - mu1);
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float al0 = up0 ? ex2_ftz(m_run[nt][0] - mu0) : 1.f;  // 2^-inf = 0 on the first keys
          const float al1 = up1 ? ex2_ftz(m_run[nt][1] - mu1) : 1.f;
          l_run[nt][0] *= al0;
          l_run[nt][1] *= al1;
          if constexpr (QK == 1) {
            psum[nt][0] *= al0;
            psum[nt][1] *= al1;
            psum[nt][2] *= al0;
            psum[nt][3] *= al1;
          }
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt) {
            o[nt][mt][0] *= al0;
            o[nt][mt][1] *= al1;
            o[nt][mt][2] *= al0;
            o[nt][mt][3] *= al1;
          }
        }
        l_run[nt][0] += p0 + p2;
        l_run[nt][1] += p1 + p3;
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
        // a value's scale multiplies its probabilities before P.V (the sums above stay unscaled)
        if constexpr (QK == 0) {
          pb[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));  // keys 0-7
          pb[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));  // keys 8-15
        } else {
          pb[nt][0] = movmatrix_trans(pack_f16x2(p0 * vs_a, p1 * vs_a));
          pb[nt][1] = movmatrix_trans(pack_f16x2(p2 * vs_b, p3 * vs_b));
        }
      }
      // O^T[d x rows] += V^T . P^T
#pragma unroll
      for (int mt = 0; mt < C::kMT; ++mt) {
        uint32_t a[4];
        if constexpr (QK == 0) {
          const int dch = mt >> 2;
          const int unit_idx = 2 * (mt & 3) + v_unit;
          ldsm_x4_trans(a, smem_addr(vt + dch * kRegionStride + swz128(v_key, unit_idx)));
        } else if constexpr (QK == 1) {  // the same, biased codes
          const uint32_t w0 = vw[mt][0] ^ 0x80808080u, w1 = vw[mt][1] ^ 0x80808080u;
          a[0] = biased2_to_f16x2(w0, kSelB02);
          a[1] = biased2_to_f16x2(w0, kSelB13);
          a[2] = biased2_to_f16x2(w1, kSelB02);
          a[3] = biased2_to_f16x2(w1, kSelB13);
        } else {  // rows g, g+8 = dims 2g, 2g+1 of the block x keys (2t, 2t+1 | 2t+8, 2t+9)
          a[0] = codes2_to_f16x2<QK>(vw[mt][0], kSelB02);
          a[1] = codes2_to_f16x2<QK>(vw[mt][0], kSelB13);
          a[2] = codes2_to_f16x2<QK>(vw[mt][1], kSelB02);
          a[3] = codes2_to_f16x2<QK>(vw[mt][1], kSelB13);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_cache<QK>(o[nt][mt], a, pb[nt][0], pb[nt][1]);
      }
      if constexpr (QK == 1) {  // the same probabilities against all-ones rows: their column sums
        const uint32_t ones[4] = {kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816_f16(psum[nt], ones, pb[nt][0], pb[nt][1]);
      }
      if constexpr (QK == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
    }
    if constexpr (QK == 1) {  // the biased values' offset
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[nt][mt][e] -= kCodeBias * psum[nt][e];
    }
    // full row sums: the 8 threads of a row each hold a share of l
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], off);
    // hand the state to the merge (the ring is free once every consumer is past its loop)
    asm volatile("bar.sync 1, %0;" ::"n"(C::kConsumers * 32));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = nt * 8 + 2 * t4 + j;
        if (g4 == 0) {
          merge_ml[(warp * ROWS + n) * 2] = m_run[nt][j];
          merge_ml[(warp * ROWS + n) * 2 + 1] = l_run[nt][j];
        }
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          // accumulator rows g, g+8: dims g, g+8 (bf16) or 2g, 2g+1 (codes) of the block
          const int d_lo = QK ? 2 * g4 : g4, d_hi = QK ? 2 * g4 + 1 : g4 + 8;
          merge_o[(warp * ROWS + n) * D + mt * 16 + d_lo] = o[nt][mt][j];
          merge_o[(warp * ROWS + n) * D + mt * 16 + d_hi] = o[nt][mt][2 + j];
        }
      }
    }
  }
  __syncthreads();
  // every CTA of the grid past its key loop lets a combine launched with programmatic stream
  // serialisation start its launch (it waits for this grid's completion before reading)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (s_timeout && threadIdx.x == C::kConsumers * 32) {
    // wind down: let copies still in flight land before the CTA's shared memory is released
    // chunk i went out iff its producer (i mod kProducers) got past it
    int hi = 0;
    for (int w = 0; w < C::kProducers; ++w) hi = max(hi, s_issued[w]);
    for (int i = max(0, hi - C::kStages); i < hi; ++i)
      if (i < s_issued[i % C::kProducers]) (void)mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1);
  }
  __syncthreads();
  merge_and_store<__nv_bfloat16>(p, merge_o, merge_ml, C::kConsumers, ROWS, D, unit, u, kvh, split);
  if (waits_for_previous) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ fp32 CUDA-core decode
// Lanes take keys for the scores (each lane one key, the group's query rows broadcast from
// shared memory) and head-dim columns for P.V. fp32 throughout, no TF32.
template <int D, int GP>
struct F32Cfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kSmemBytes =
      (GP * D + kWarps * GP * 32 + kWarps * GP * D + kWarps * GP * 2) * 4 + kWarps * 32 * 8;
};

template <int D, int GP>
__global__ void __launch_bounds__(128) decode_f32_kernel(const __grid_constant__ DecodeParams p) {
  using C = F32Cfg<D, GP>;
  constexpr int DL = D / 32;  // columns per lane
  extern __shared__ float fsm[];
  float* q_s = fsm;                               // [GP][D]
  float* p_s = q_s + GP * D;                      // [warps][GP][32]
  float* merge_o = p_s + C::kWarps * GP * 32;     // [warps][GP][D]
  float* merge_ml = merge_o + C::kWarps * GP * D; // [warps][GP][2]
  long long* vrow_s = reinterpret_cast<long long*>(merge_ml + C::kWarps * GP * 2);  // [warps][32]

  const int unit = blockIdx.x / p.num_splits;
  const int split = blockIdx.x - unit * p.num_splits;
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const Unit u = resolve_unit(p, unit, threadIdx.x == 0 && split == 0 && kvh == 0);
  if (u.skip) return;
  const int k_begin = max(split * p.chunks_per_split * kChunk, u.start);
  const int k_end = min(u.len, split * p.chunks_per_split * kChunk + p.chunks_per_split * kChunk);

  const float* qg = reinterpret_cast<const float*>(p.q) + (size_t)u.q_row * p.q_stride + (size_t)kvh * G * D;
  for (int idx = threadIdx.x; idx < GP * D; idx += blockDim.x) q_s[idx] = (idx / D < G) ? qg[idx] : 0.f;
  __syncthreads();

  const float* kc = reinterpret_cast<const float*>(p.k_cache);
  const float* vc = reinterpret_cast<const float*>(p.v_cache);
  const int32_t* table = p.block_tables + (size_t)u.table_row * p.max_blocks;
  const size_t row_elems = (size_t)p.num_kv_heads * D;
  float m_run[GP], l_run[GP], acc[GP][DL];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.f;
#pragma unroll
    for (int j = 0; j < DL; ++j) acc[g][j] = 0.f;
  }
  float* my_p = p_s + warp * GP * 32;
  long long* my_vrow = vrow_s + warp * 32;
  for (int kb = k_begin + warp * 32; kb < k_end; kb += C::kWarps * 32) {
    const int key = kb + lane;
    const bool valid = key < k_end;
    long long row = 0;
    if (valid) {
      int page = table[key / p.block_size];
      if (page < 0 || page >= p.num_blocks) {
        flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);
        page = -1;
      }
      row = (page < 0) ? -1 : ((long long)page * p.block_size + key % p.block_size);
    }
    float s[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) s[g] = 0.f;
    if (valid && row >= 0) {
      const float4* kr = reinterpret_cast<const float4*>(kc + (size_t)row * row_elems + (size_t)kvh * D);
#pragma unroll 8
      for (int d4 = 0; d4 < D / 4; ++d4) {
        const float4 k4 = __ldg(kr + d4);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float4 q4 = reinterpret_cast<const float4*>(q_s + g * D)[d4];
          s[g] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, s[g]))));
        }
      }
    }
    my_vrow[lane] = valid ? row : -2;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float x = valid ? score_log2(p, s[g]) : -INFINITY;
      float mx = x;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m_run[g], mx);
      const float mu = (mn == -INFINITY) ? 0.f : mn;
      const float al = exp2f(m_run[g] - mu);
      const float pr = valid ? exp2f(x - mu) : 0.f;
      l_run[g] = l_run[g] * al + pr;
      m_run[g] = mn;
#pragma unroll
      for (int j = 0; j < DL; ++j) acc[g][j] *= al;
      my_p[g * 32 + lane] = pr;
    }
    __syncwarp();
    // value rows in batches whose loads are all issued before the first is used (one memory
    // latency per batch, not per key); a row past the end or outside the pool reads as zeros
    // and its probability is 0
    const int nk = min(32, k_end - kb);
    constexpr int kVB = DL >= 8 ? 4 : 8;
    for (int j0 = 0; j0 < nk; j0 += kVB) {
      float vv[kVB][DL];
#pragma unroll
      for (int b = 0; b < kVB; ++b) {
        const long long vr = j0 + b < nk ? my_vrow[j0 + b] : -1;
        const float* vrp = vc + (size_t)(vr < 0 ? 0 : vr) * row_elems + (size_t)kvh * D;
#pragma unroll
        for (int c = 0; c < DL; ++c) vv[b][c] = vr >= 0 ? __ldg(vrp + lane + 32 * c) : 0.f;
      }
#pragma unroll
      for (int b = 0; b < kVB; ++b) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pj = my_p[g * 32 + j0 + b];
#pragma unroll
          for (int c = 0; c < DL; ++c) acc[g][c] = fmaf(pj, vv[b][c], acc[g][c]);
        }
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int g = 0; g < GP; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], off);
    if (lane == 0) {
      merge_ml[(warp * GP + g) * 2] = m_run[g];
      merge_ml[(warp * GP + g) * 2 + 1] = l_run[g];
    }
#pragma unroll
    for (int c = 0; c < DL; ++c) merge_o[(warp * GP + g) * D + lane + 32 * c] = acc[g][c];
  }
  __syncthreads();
  merge_and_store<float>(p, merge_o, merge_ml, C::kWarps, GP, D, unit, u, kvh, split);
}

// ------------------------------------------------------------------ combine
// One warp per (unit, query head): M = max_s m_s, w_s = 2^(m_s - M),
// out = sum_s w_s acc_s / sum_s w_s l_s; an all-empty row (M = -inf) gives zeros.
// ("32. Production attention kernels", Long contexts: split the keys, the merge;
//  "poot - Attention and KV Cache", Split-KV decode, Combine.)
template <typename OutT>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ DecodeParams p) {
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int T = p.unit_tokens;  // queries per unit
  if (gw >= p.num_units * T * p.num_q_heads) return;
  // launched as a programmatic dependent of the split kernel: wait for that grid to complete
  // and its partials to be visible (a no-op for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int unit = gw / (T * p.num_q_heads);
  const int rem = gw - unit * T * p.num_q_heads;
  const int t = rem / p.num_q_heads;  // query t of the unit
  const int h = rem - t * p.num_q_heads;
  const int S = p.num_splits;
  // the row's output row (request units: only the queries the split kernel served)
  int q_row = unit;
  if (p.varlen == 2) {
    const int r = unit / p.groups_per_req;
    const int tok = (unit - r * p.groups_per_req) * T + t;
    const int start = p.query_start_loc[r];
    const int q_len = p.query_start_loc[r + 1] - start;
    if (start < 0 || q_len < 1 || q_len > p.small_max || tok >= q_len || start + q_len > p.num_tokens) return;
    q_row = start + tok;
  }
  const int D = p.head_dim;
  const size_t sstride = (size_t)T * p.num_q_heads;       // slot of split s: base + s * sstride
  const size_t base = (size_t)unit * S * sstride + (size_t)t * p.num_q_heads + h;
  // Sixteen partials' loads per batch are issued before any of them is used, so their latencies
  // overlap; the first batch is requested before the weights, so it overlaps the (m, l) loads too.
  constexpr int kBatch = 8;
  auto load_batch = [&](int d0, int s0, float4 (&v)[kBatch]) {
    const int d = d0 + lane * 4;
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      v[k] = (d < D && s0 + k < S)
                 ? *reinterpret_cast<const float4*>(p.ws_acc + (base + (size_t)(s0 + k) * sstride) * D + d)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  float4 first[kBatch];
  load_batch(0, 0, first);
  const float m_s = (lane < S) ? p.ws_ml[(base + (size_t)lane * sstride) * 2] : -INFINITY;
  const float l_s = (lane < S) ? p.ws_ml[(base + (size_t)lane * sstride) * 2 + 1] : 0.f;
  float M = m_s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  // a sink logit joins the denominator here, once, not in every split
  const float z2 = p.sinks != nullptr ? p.sinks[h] * kLog2e : -INFINITY;
  M = fmaxf(M, z2);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  const float w = (lane < S) ? exp2f(m_s - Mu) : 0.f;
  float L = w * l_s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  L += exp2f(z2 - Mu);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  OutT* out = reinterpret_cast<OutT*>(p.out) + (size_t)q_row * p.out_stride + (size_t)h * D;
  // every lane runs every iteration (the weight shuffles need the whole warp); lanes past
  // the head dim only skip their loads and stores
  for (int d0 = 0; d0 < D; d0 += 128) {
    const int d = d0 + lane * 4;
    const bool active = d < D;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += kBatch) {
      float4 v[kBatch];
      if (d0 == 0 && s0 == 0) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k) v[k] = first[k];
      } else {
        load_batch(d0, s0, v);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float ws = __shfl_sync(0xffffffffu, w, (s0 + k) & 31);  // w = 0 on lanes >= S
        a.x = fmaf(ws, v[k].x, a.x);
        a.y = fmaf(ws, v[k].y, a.y);
        a.z = fmaf(ws, v[k].z, a.z);
        a.w = fmaf(ws, v[k].w, a.w);
      }
    }
    if (active) {
      out[d] = static_cast<OutT>(a.x * inv);
      out[d + 1] = static_cast<OutT>(a.y * inv);
      out[d + 2] = static_cast<OutT>(a.z * inv);
      out[d + 3] = static_cast<OutT>(a.w * inv);
    }
  }
}

template <int D, int NT, int QK>
cudaError_t launch_tc_impl(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
  using C = DecCfg<D, QK>;
  auto kern = decode_tc_kernel<D, NT, QK>;
  // the shared-memory opt-in is per device; setting it again is harmless, so concurrent first
  // calls from several host threads may both set it
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  dim3 grid((unsigned)(p.num_units * p.num_splits), (unsigned)p.num_kv_heads, 1);
  if (!p.overlap_previous) {
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(p, kmap, vmap);
    return cudaGetLastError();
  }
  // programmatic dependent launch: the CTAs may start while the previous kernel still runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, kmap, vmap);
}

template <int D, int NT, int QK>
int occupancy_tc() {
  using C = DecCfg<D, QK>;
  auto kern = decode_tc_kernel<D, NT, QK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::kSmemBytes) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

template <int D, int GP>
cudaError_t launch_f32_impl(const DecodeParams& p, cudaStream_t stream) {
  using C = F32Cfg<D, GP>;
  auto kern = decode_f32_kernel<D, GP>;
  if (C::kSmemBytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)(p.num_units * p.num_splits), (unsigned)p.num_kv_heads, 1);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int GP>
int occupancy_f32() {
  using C = F32Cfg<D, GP>;
  auto kern = decode_f32_kernel<D, GP>;
  if (C::kSmemBytes > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::kThreads, C::kSmemBytes) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

int pad_group(int g) {
  int gp = 1;
  while (gp < g) gp <<= 1;
  return gp;
}

// q / out row strides default to dense rows; units default to one query
DecodeParams with_row_strides(const DecodeParams& in) {
  DecodeParams p = in;
  if (p.q_stride == 0) p.q_stride = (long long)p.num_q_heads * p.head_dim;
  if (p.out_stride == 0) p.out_stride = (long long)p.num_q_heads * p.head_dim;
  if (p.unit_tokens < 1) p.unit_tokens = 1;
  if (p.groups_per_req < 1) p.groups_per_req = 1;
  return p;
}

}  // namespace

// one n-tile of 8 rows, or two for up to 16 rows (rows = unit queries x group)
#define PA_TC_NT(D, QK)                                                                 \
  (p.unit_tokens * p.group > 8 ? launch_tc_impl<D, 2, QK>(p, kmap, vmap, stream)        \
                               : launch_tc_impl<D, 1, QK>(p, kmap, vmap, stream))

cudaError_t launch_decode_bf16(const DecodeParams& p_in, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t stream) {
  const DecodeParams p = with_row_strides(p_in);
  switch (p.quant * 1000 + p.head_dim) {
    case 64: return PA_TC_NT(64, 0);
    case 128: return PA_TC_NT(128, 0);
    case 256: return PA_TC_NT(256, 0);
    case 1128: return PA_TC_NT(128, 1);
    case 1256: return PA_TC_NT(256, 1);
    case 2128: return PA_TC_NT(128, 2);
    case 2256: return PA_TC_NT(256, 2);
    default: return cudaErrorInvalidValue;
  }
}

#define PA_TC_OCC(D, QK) (group > 8 ? occupancy_tc<D, 2, QK>() : occupancy_tc<D, 1, QK>())

int decode_bf16_ctas_per_sm(int head_dim, int group, int quant) {
  switch (quant * 1000 + head_dim) {
    case 64: return PA_TC_OCC(64, 0);
    case 128: return PA_TC_OCC(128, 0);
    case 256: return PA_TC_OCC(256, 0);
    case 1128: return PA_TC_OCC(128, 1);
    case 1256: return PA_TC_OCC(256, 1);
    case 2128: return PA_TC_OCC(128, 2);
    case 2256: return PA_TC_OCC(256, 2);
    default: return 1;
  }
}

#define PA_F32_CASES(D)                                         \
  switch (pad_group(p.group)) {                                 \
    case 1: return launch_f32_impl<D, 1>(p, stream);            \
    case 2: return launch_f32_impl<D, 2>(p, stream);            \
    case 4: return launch_f32_impl<D, 4>(p, stream);            \
    case 8: return launch_f32_impl<D, 8>(p, stream);            \
    case 16: if (D <= 128) return launch_f32_impl<(D <= 128 ? D : 128), 16>(p, stream); \
             return cudaErrorInvalidValue;                      \
    default: return cudaErrorInvalidValue;                      \
  }

cudaError_t launch_decode_f32(const DecodeParams& p_in, cudaStream_t stream) {
  const DecodeParams p = with_row_strides(p_in);
  switch (p.head_dim) {
    case 64: PA_F32_CASES(64)
    case 128: PA_F32_CASES(128)
    case 256: PA_F32_CASES(256)
    default: return cudaErrorInvalidValue;
  }
}

#define PA_F32_OCC(D)                                           \
  switch (pad_group(group)) {                                   \
    case 1: return occupancy_f32<D, 1>();                       \
    case 2: return occupancy_f32<D, 2>();                       \
    case 4: return occupancy_f32<D, 4>();                       \
    case 8: return occupancy_f32<D, 8>();                       \
    case 16: return occupancy_f32<(D <= 128 ? D : 128), 16>();  \
    default: return 1;                                          \
  }

int decode_f32_ctas_per_sm(int head_dim, int group) {
  switch (head_dim) {
    case 64: PA_F32_OCC(64)
    case 128: PA_F32_OCC(128)
    case 256: PA_F32_OCC(256)
    default: return 1;
  }
}

cudaError_t launch_combine(const DecodeParams& p_in, pa_dtype dtype, cudaStream_t stream) {
  const DecodeParams p = with_row_strides(p_in);
  const long long warps = (long long)p.num_units * p.unit_tokens * p.num_q_heads;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  // programmatic dependent launch: the combine's CTAs launch while the split kernel's last CTAs
  // merge and store, and wait in-kernel for its completion
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == PA_DTYPE_BF16) return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, p);
}

}  // namespace pa
